"""No write lands outside the output: the output (and, in the fp32 mode, the
index output) sits inside a larger buffer whose guard regions before and
after it hold a sentinel, and the sentinel must survive the forward.  The
shapes are the ragged ones: odd output widths, padded channel tiles, the
column-tiled rows, the atomic-minimum channel tiles (whose output is filled
with +inf first), and the GroupNorm chain's float4 finalize stores.  The
result inside the guards must still match the oracle.  Collected near the
end of the suite, after the parity tests."""
import numpy as np
import pytest

import oracle
import synth
from parity_util import check_fp32, check_tf32, epilogue_for, oracle_run, torch_inputs

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
CASES = {
    "c2_w255": W["c2_min_tanh2"].resized(N=1, H=7, W=255),                # odd output rows, padded input rows
    "c3_w67": W["c3_mul_lrelu_gelu"].resized(N=2, H=6, W=67),            # per-channel scalar stores
    "c3_co200": W["c3_mul_lrelu_gelu"].resized(N=1, H=5, W=64, Cout=200),  # second channel tile padded
    "c4_co256": W["c4_scale_min"].resized(N=1, H=5, W=64, Cout=256),     # output fill, atomic minimum
    "c4_w516": W["c4_scale_min"].resized(N=2, H=4, W=516, scalar=-1.0),  # three column tiles
    "c5t": W["c5_gn_pool_clamp"].resized(N=2, H=40),                     # pooled rows past the last band
    "c5_w37": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=37),            # two bands, columns past the pool
    "min_cout1": W["pr1_min_tanh2"].resized(N=1, Cin=1, H=3, W=4, Cout=1),
    # narrow rows with many output channels: the fp32 kernel stages fewer
    # channel slots per pass so the filter taps fit shared memory
    "c4_co512_w8": W["c4_scale_min"].resized(N=2, H=6, W=8, Cout=512),
    "c3_co640_w10": W["c3_mul_lrelu_gelu"].resized(N=1, Cin=24, H=5, W=10, Cout=640),
    # the plain conv output: 16-byte row stores where rows start aligned
    # (ragged last float4 of 254- and 62-wide rows), 8-byte or single-float
    # stores elsewhere
    "none_w256": W["c3_mul_lrelu_gelu"].resized(N=1, H=6, kind=synth.KIND_NONE),
    "none_w64": W["c3_mul_lrelu_gelu"].resized(N=2, H=7, W=64, Cout=40, kind=synth.KIND_NONE),
    "none_w67": W["c3_mul_lrelu_gelu"].resized(N=1, H=6, W=67, kind=synth.KIND_NONE),
    "none_w520_co200": W["c3_mul_lrelu_gelu"].resized(N=1, H=4, W=520, Cout=200, kind=synth.KIND_NONE),
}
GUARD = 64          # elements on each side (256 bytes: the output stays 16-byte aligned)
SENTINEL = -1234.5
ISENTINEL = -99


def guarded(shape, dtype, fill):
    import torch
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * GUARD,), fill, dtype=dtype, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(shape)


def guards_intact(buf, n, fill):
    b = buf.cpu().numpy()
    return bool(np.all(b[:GUARD] == fill) and np.all(b[GUARD + n:] == fill))


@pytest.mark.parametrize("mode", ["tf32", "fp32"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_writes_stay_inside_the_output(case, mode):
    import torch
    import x3_conv2d_epilogue_gb300 as ce
    wl = CASES[case]
    m = ce.MODE_TF32 if mode == "tf32" else ce.MODE_FP32
    t = synth.make_inputs(wl, seed=5)
    d = torch_inputs(t)
    probe = ce.epilogue(wl.kind, groups=wl.groups, pool_k=wl.pool_k, chan_scale=1, gamma=1, beta=1)
    shape = ce.conv_epi_output_shape(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, probe, m)
    n = int(np.prod(shape))
    obuf, out = guarded(shape, torch.float32, SENTINEL)
    ibuf, idx = (None, None)
    if m == ce.MODE_FP32 and wl.kind not in (synth.KIND_MUL_LRELU_GELU, synth.KIND_NONE):
        ibuf, idx = guarded(shape, torch.int32, ISENTINEL)
    epi = epilogue_for(wl, d, idx)
    h = ce.conv_epi_create(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, m)
    try:
        ce.conv_epi_forward(h, d["x"], d["w"], d["b"], epi, out)
        ce.conv_epi_sync(h)
    finally:
        ce.conv_epi_destroy(h)
    torch.cuda.synchronize()
    assert guards_intact(obuf, n, SENTINEL), f"{case} {mode}: a write landed outside the output"
    if ibuf is not None:
        assert guards_intact(ibuf, n, ISENTINEL), f"{case} {mode}: a write landed outside the index output"
    ref = oracle.conv3x3(t.x, t.w, t.b) if wl.kind == synth.KIND_NONE else oracle_run(wl, t)[0]
    got = out.cpu().numpy()
    if m == ce.MODE_FP32:
        check_fp32(got, ref, case)
    else:
        check_tf32(got, ref, case)


@pytest.mark.parametrize("mode", ["tf32", "fp32"])
def test_empty_batch_is_a_no_op(mode):
    """N = 0: a handle is created, every forward (device and host buffers,
    every chain) returns OK with empty tensors and launches nothing."""
    import torch
    import x3_conv2d_epilogue_gb300 as ce
    m = ce.MODE_TF32 if mode == "tf32" else ce.MODE_FP32
    p = torch.ones(64, device="cuda")
    chains = [ce.epilogue(ce.MIN_TANH2), ce.epilogue(ce.SCALE_MIN, scalar=-2.0),
              ce.epilogue(ce.MUL_LRELU_GELU, chan_scale=p),
              ce.epilogue(ce.GN_SCALE_POOL_CLAMP, chan_scale=p, gamma=p, beta=p, groups=16, pool_k=4),
              ce.epilogue(ce.NONE)]
    x = torch.empty(0, 8, 18, 16, device="cuda")
    w = torch.zeros(64, 8, 3, 3, device="cuda")
    h = ce.conv_epi_create(0, 8, 18, 16, 64, m)
    try:
        for epi in chains:
            out = torch.empty(ce.conv_epi_output_shape(0, 8, 18, 16, 64, epi, m), device="cuda")
            assert out.numel() == 0
            ce.conv_epi_forward(h, x, w, p, epi, out)
            assert ce.conv_epi_last_launch_count(h) == 0
        ce.conv_epi_sync(h)
        host = ce.epilogue(ce.MIN_TANH2)
        ce.conv_epi_forward_host(h, np.empty((0, 8, 18, 16), np.float32), np.zeros((64, 8, 3, 3), np.float32),
                                 np.ones(64, np.float32), host, np.empty((0, 1, 16, 14), np.float32))
    finally:
        ce.conv_epi_destroy(h)
