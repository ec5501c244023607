"""GPU parity at the full workload sizes, in the launch configuration the
bench times: the whole batch in one conv_epi_forward, both modes (tf32 also with
channels-last input).  The oracle
checks sampled outputs one by one (min chains: whole channel columns;
per-channel chain: single elements; GroupNorm chain: every pooled output of
a few whole (image, group) pairs, statistics included), and properties that
hold at every output (finite; tanh∘tanh inside (-tanh 1, tanh 1); clamp range).
In fp32 mode the reductions' indices are checked too (channel of the
minimum, window offset of the pooled value): at the sampled points, and over
the whole first and last images element by element, exact wherever the
oracle's best and second-best candidates differ by more than 1e-5.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from parity_util import (FP32_ATOL, TF32_ATOL, TF32_RTOL, check_fp32, check_index, epilogue_for, min_index_gap,
                         pool_index_gap, torch_inputs)

pytestmark = pytest.mark.gpu

NS = 256          # sampled outputs per check
GN_GROUPS = 3     # (n, g) pairs checked for the GroupNorm chain


@pytest.fixture(scope="module", params=["c2_min_tanh2", "c3_mul_lrelu_gelu", "c4_scale_min", "c5_gn_pool_clamp"])
def full(request):
    wl = synth.WORKLOADS[request.param]
    t = synth.make_inputs(wl, seed=0)
    return wl, t, torch_inputs(t)


def run(wl, d, mode, layout=0, want_index=False):
    """One forward over the whole batch; (out, index or None) as torch tensors."""
    import torch
    import x3_conv2d_epilogue_gb300 as ce
    probe = epilogue_for(wl, d)
    shape = ce.conv_epi_output_shape(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, probe, mode)
    idx = torch.full(shape, -7, device="cuda", dtype=torch.int32) if want_index else None
    epi = epilogue_for(wl, d, idx)
    x = d["x"].permute(0, 2, 3, 1).contiguous() if layout == ce.LAYOUT_NHWC else d["x"]
    h = ce.conv_epi_create(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, mode, layout)
    try:
        out = torch.full(shape, float("nan"), device="cuda", dtype=torch.float32)
        ce.conv_epi_forward(h, x, d["w"], d["b"], epi, out)
        ce.conv_epi_sync(h)
    finally:
        ce.conv_epi_destroy(h)
    return out, idx


def close(got, ref, mode):
    err = np.abs(got.astype(np.float64) - ref)
    if mode == "fp32":
        return err <= FP32_ATOL, err
    return err <= TF32_ATOL + TF32_RTOL * np.abs(ref), err


@pytest.mark.parametrize("mode", ["tf32", "fp32", "tf32_nhwc"])
def test_full_size(full, mode):
    import torch
    import x3_conv2d_epilogue_gb300 as ce
    wl, t, d = full
    m = ce.MODE_FP32 if mode == "fp32" else ce.MODE_TF32
    out, _ = run(wl, d, m, ce.LAYOUT_NHWC if mode == "tf32_nhwc" else ce.LAYOUT_NCHW)
    mode = "fp32" if mode == "fp32" else "tf32"  # the tolerance
    assert bool(torch.isfinite(out).all()), "non-finite outputs"
    rng = np.random.default_rng(1234)
    Ho, Wo = wl.H - 2, wl.W - 2
    if wl.kind in (synth.KIND_MIN_TANH2, synth.KIND_SCALE_MIN):
        if wl.kind == synth.KIND_MIN_TANH2:
            assert float(out.abs().max()) < math.tanh(1.0)
        n, i, j = rng.integers(0, wl.N, NS), rng.integers(0, Ho, NS), rng.integers(0, Wo, NS)
        # always include the image corners and the last rows/columns
        n[:4], i[:4], j[:4] = [0, wl.N - 1, 0, wl.N - 1], [0, Ho - 1, Ho - 1, 0], [0, Wo - 1, 0, Wo - 1]
        ref, _ = oracle.min_at(t.x, t.w, t.b, n, i, j, scalar=wl.scalar, tanh2=wl.kind == synth.KIND_MIN_TANH2)
        idx = torch.as_tensor(np.stack([n, np.zeros_like(n), i, j]), device="cuda")
        got = out[idx[0], idx[1], idx[2], idx[3]].cpu().numpy()
    elif wl.kind == synth.KIND_MUL_LRELU_GELU:
        n, co = rng.integers(0, wl.N, NS), rng.integers(0, wl.Cout, NS)
        i, j = rng.integers(0, Ho, NS), rng.integers(0, Wo, NS)
        n[:2], co[:2], i[:2], j[:2] = [0, wl.N - 1], [0, wl.Cout - 1], [0, Ho - 1], [0, Wo - 1]
        ref = oracle.mul_lrelu_gelu_at(t.x, t.w, t.b, t.mult, n, co, i, j, slope=wl.lrelu_slope)
        got = out[torch.as_tensor(n), torch.as_tensor(co), torch.as_tensor(i), torch.as_tensor(j)].cpu().numpy()
    else:
        assert float(out.min()) >= wl.clamp_lo and float(out.max()) <= wl.clamp_hi
        ch = oracle.chain_for(wl, t)
        cpg = wl.Cout // wl.groups
        pairs = [(0, 0), (wl.N - 1, wl.groups - 1)] + [(int(rng.integers(0, wl.N)), int(rng.integers(0, wl.groups)))
                                                       for _ in range(GN_GROUPS - 2)]
        refs, gots = [], []
        for (n, g) in pairs:
            r, _, _, _ = oracle.gn_group(t.x, t.w, t.b, ch, n, g)
            refs.append(r.ravel())
            gots.append(out[n, g * cpg:(g + 1) * cpg].cpu().numpy().ravel())
        ref, got = np.concatenate(refs), np.concatenate(gots)
    ok, err = close(got, ref, mode)
    assert ok.all(), f"{wl.name} {mode}: {int((~ok).sum())} of {ok.size} sampled outputs off; max err {err.max():.3g}"


def gap_at_points(t, wl, n, i, j):
    """Best-vs-second gap of scalar * y over the channels at sampled points."""
    y = np.array([[oracle.conv_at(t.x, t.w, t.b, int(a), co, int(p), int(q)) for co in range(wl.Cout)]
                  for a, p, q in zip(n, i, j)])
    v = np.sort(wl.scalar * y, axis=1)
    return v[:, 1] - v[:, 0]


@pytest.mark.parametrize("wl_name", ["c2_min_tanh2", "c4_scale_min", "c5_gn_pool_clamp"])
def test_full_size_fp32_indices(wl_name):
    """fp32 mode at full size with the index output: values and indices of
    the first and last whole images against the oracle's forward on those
    images, plus (min chains) 256 sampled points across the batch."""
    import x3_conv2d_epilogue_gb300 as ce
    wl = synth.WORKLOADS[wl_name]
    t = synth.make_inputs(wl, seed=0)
    d = torch_inputs(t)
    out, idx = run(wl, d, ce.MODE_FP32, want_index=True)
    ties = 0
    for img in (0, wl.N - 1):
        one = wl.with_batch(1)
        ti = synth.Tensors(t.x[img:img + 1], t.w, t.b, t.mult, t.gamma, t.beta, t.scale)
        ref, ref_idx = oracle.forward(ti.x, ti.w, ti.b, oracle.chain_for(one, ti))
        got, got_idx = out[img:img + 1].cpu().numpy(), idx[img:img + 1].cpu().numpy()
        check_fp32(got, ref, f"{wl_name} image {img}")
        y = oracle.conv3x3(ti.x, ti.w, ti.b)
        if wl.kind == synth.KIND_GN_SCALE_POOL_CLAMP:
            slope = t.gamma.astype(np.float64) * t.scale
            gap = pool_index_gap(y, wl.pool_k, np.where(slope >= 0, 1.0, -1.0)[None, :]) * np.abs(slope)[None, :, None, None]
        else:
            gap = min_index_gap(y, wl.scalar)
        ties += check_index(got_idx, ref_idx, gap, f"{wl_name} image {img}")
    if wl.kind != synth.KIND_GN_SCALE_POOL_CLAMP:
        rng = np.random.default_rng(99)
        Ho, Wo = wl.H - 2, wl.W - 2
        n, i, j = rng.integers(0, wl.N, NS), rng.integers(0, Ho, NS), rng.integers(0, Wo, NS)
        _, ref_idx = oracle.min_at(t.x, t.w, t.b, n, i, j, scalar=wl.scalar, tanh2=wl.kind == synth.KIND_MIN_TANH2)
        got_idx = idx.cpu().numpy()[n, 0, i, j]
        ties += check_index(got_idx, ref_idx, gap_at_points(t, wl, n, i, j), f"{wl_name} sampled")
    assert ties <= 16, f"{ties} near-tie index differences"


# GroupNorm shapes beyond the page's, at the page's batch and image size (the
# generalised kernel instantiations, whose finalize runs a ring of pair
# slots that turns over several times per CTA): every pooled output of a few
# whole (image, group) pairs against the oracle, among them the pairs that
# land in the ring's last slots
GN_WIDE = {
    "c5_pool2": synth.WORKLOADS["c5_gn_pool_clamp"].resized(pool_k=2),                 # 2x2 windows
    "c5_co128": synth.WORKLOADS["c5_gn_pool_clamp"].resized(Cout=128, groups=16),      # half bands
    "c5_w256": synth.WORKLOADS["c5_gn_pool_clamp"].resized(N=32, H=256, W=256),        # wide rows
    "c5_co256": synth.WORKLOADS["c5_gn_pool_clamp"].resized(Cout=256, groups=32),     # channel tiles
    "c5_w512": synth.WORKLOADS["c5_gn_pool_clamp"].resized(N=8, H=512, W=512),         # column tiles, separate finalize
    "c5_pool2_co128": synth.WORKLOADS["c5_gn_pool_clamp"].resized(Cout=128, groups=16, pool_k=2),  # 2x2, no stacking
    "c5_pool2_w64": synth.WORKLOADS["c5_gn_pool_clamp"].resized(N=256, H=64, W=64, pool_k=2),      # 2x2, four bands per unit
    "c5_pool2_w240": synth.WORKLOADS["c5_gn_pool_clamp"].resized(N=32, H=240, W=240, pool_k=2),    # 2x2, rows of 238
    "c5_co128_w256": synth.WORKLOADS["c5_gn_pool_clamp"].resized(N=32, H=256, W=256, Cout=128, groups=16),  # quarter bands
}


@pytest.mark.parametrize("case", sorted(GN_WIDE))
def test_full_batch_generalised_groupnorm(case):
    import x3_conv2d_epilogue_gb300 as ce
    wl = GN_WIDE[case]
    t = synth.make_inputs(wl, seed=0)
    out, _ = run(wl, torch_inputs(t), ce.MODE_TF32)
    import torch
    assert bool(torch.isfinite(out).all()), "non-finite outputs"
    assert float(out.min()) >= wl.clamp_lo and float(out.max()) <= wl.clamp_hi
    ch = oracle.chain_for(wl, t)
    cpg = wl.Cout // wl.groups
    npairs = wl.N * wl.groups
    # pair p is finalized by CTA p % 152 as its (p // 152)-th pair
    picks = [0, npairs - 1, min(npairs - 1, 12 * 152 + 5), min(npairs - 1, 7 * 152 + 100)]
    refs, gots = [], []
    for p in picks:
        n, g = divmod(p, wl.groups)
        r, _, _, _ = oracle.gn_group(t.x, t.w, t.b, ch, n, g)
        refs.append(r.ravel())
        gots.append(out[n, g * cpg:(g + 1) * cpg].cpu().numpy().ravel())
    ref, got = np.concatenate(refs), np.concatenate(gots)
    ok, err = close(got, ref, "tf32")
    assert ok.all(), f"{case}: {int((~ok).sum())} of {ok.size} outputs off; max err {err.max():.3g}"
