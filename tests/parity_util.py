"""Helpers shared by the parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs, compare within the stated bounds.

Tolerances (stated for the method's two arithmetic modes):
  fp32 CUDA-core mode : max |gpu - oracle| <= 1e-4, indices exact where the
                        oracle's best and second-best candidates differ by
                        more than 1e-5 (nearer ties are counted, not failed);
  tf32 tensor mode    : |gpu - oracle| <= 5e-3 + 5e-3 * |oracle| everywhere.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth

FP32_ATOL = 1e-4
TF32_ATOL = 5e-3
TF32_RTOL = 5e-3
TIE_GAP = 1e-5


def torch_inputs(t: synth.Tensors, device="cuda"):
    import torch
    d = {}
    for k in ("x", "w", "b", "mult", "gamma", "beta", "scale"):
        v = getattr(t, k)
        d[k] = None if v is None else torch.from_numpy(np.ascontiguousarray(v)).to(device)
    return d


def epilogue_for(wl: synth.Workload, d, index_out=None):
    import x3_conv2d_epilogue_gb300 as ce
    chan = d["mult"] if wl.kind == synth.KIND_MUL_LRELU_GELU else d["scale"]
    return ce.epilogue(wl.kind, scalar=wl.scalar, chan_scale=chan, lrelu_slope=wl.lrelu_slope, groups=wl.groups,
                       eps=wl.eps, gamma=d["gamma"], beta=d["beta"], pool_k=wl.pool_k, clamp_lo=wl.clamp_lo,
                       clamp_hi=wl.clamp_hi, index_out=index_out)


def fp32_indices(wl: synth.Workload) -> bool:
    """The fp32 mode returns indices for the min chains and for the GroupNorm
    chain it runs fused (pool_k 1, 2 or 4, at most 64 groups); its two-pass
    GroupNorm form (any other pool_k or group count) gives none."""
    if wl.kind == synth.KIND_MUL_LRELU_GELU or wl.kind == synth.KIND_NONE:
        return False
    return wl.kind != synth.KIND_GN_SCALE_POOL_CLAMP or (wl.pool_k in (1, 2, 4) and wl.groups <= 64)


def gpu_run(wl: synth.Workload, t: synth.Tensors, mode: int, want_index=False, repeats=1, layout=0):
    """Run conv + chain on cuda:0 through the C ABI; returns numpy (out, index).
    layout 1 hands the library x in channels-last order (a transposed copy of
    the same values)."""
    import torch
    import x3_conv2d_epilogue_gb300 as ce
    d = torch_inputs(t)
    if layout == ce.LAYOUT_NHWC:
        d["x"] = d["x"].permute(0, 2, 3, 1).contiguous()
    probe = ce.epilogue(wl.kind, groups=wl.groups, pool_k=wl.pool_k, chan_scale=1, gamma=1, beta=1)
    shape = ce.conv_epi_output_shape(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, probe, mode)
    out = torch.full(shape, float("nan"), device="cuda", dtype=torch.float32)
    idx = torch.full(shape, -7, device="cuda", dtype=torch.int32) if want_index else None
    epi = epilogue_for(wl, d, idx)
    h = ce.conv_epi_create(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, mode, layout)
    try:
        for _ in range(repeats):
            ce.conv_epi_forward(h, d["x"], d["w"], d["b"], epi, out)
        ce.conv_epi_sync(h)
    finally:
        ce.conv_epi_destroy(h)
    torch.cuda.synchronize()
    return out.cpu().numpy(), (idx.cpu().numpy() if want_index else None)


def oracle_run(wl: synth.Workload, t: synth.Tensors):
    return oracle.forward(t.x, t.w, t.b, oracle.chain_for(wl, t))


def check_fp32(got, ref, what=""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    err = np.abs(got.astype(np.float64) - ref)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= FP32_ATOL, f"{what}: max |err| {worst:.3g} > {FP32_ATOL} at {np.unravel_index(err.argmax(), err.shape)}"
    return worst


def check_tf32(got, ref, what=""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    err = np.abs(got.astype(np.float64) - ref)
    bound = TF32_ATOL + TF32_RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside 5e-3+5e-3|ref|; worst err "
                           f"{float(err.max()):.3g} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max()) if err.size else 0.0


def min_index_gap(y: np.ndarray, scalar: float) -> np.ndarray:
    """Per pixel: gap between the best and second-best channel of scalar*y."""
    v = np.sort(scalar * y, axis=1)
    return v[:, 1:2] - v[:, 0:1]


def pool_index_gap(y: np.ndarray, pool_k: int, mean_sign: np.ndarray) -> np.ndarray:
    """Per pooled output: gap between the best and second-best window entry of
    y (largest when the channel's affine slope is >= 0, smallest otherwise)."""
    N, Cc, Ho, Wo = y.shape
    Hp, Wp = (Ho - pool_k) // pool_k + 1, (Wo - pool_k) // pool_k + 1
    win = y[:, :, :Hp * pool_k, :Wp * pool_k].reshape(N, Cc, Hp, pool_k, Wp, pool_k).transpose(0, 1, 2, 4, 3, 5)
    win = win.reshape(N, Cc, Hp, Wp, pool_k * pool_k)
    win = win * mean_sign.reshape(N, Cc, 1, 1, 1)
    if pool_k == 1:     # a one-entry window: its index is the only one
        return np.full(win.shape[:-1], np.inf)
    v = np.sort(win, axis=-1)
    return v[..., -1] - v[..., -2]


def check_index(got_idx, ref_idx, gap, what=""):
    mism = (got_idx != ref_idx)
    clear = gap > TIE_GAP
    hard = mism & clear
    assert not hard.any(), f"{what}: {int(hard.sum())} index mismatches away from ties (first at {np.argwhere(hard)[0]})"
    return int((mism & ~clear).sum())
