"""conv_epi_forward_host: host buffers in, host buffers out, the batch sliced
into up to eight groups of whole images whose copies overlap the compute.
Each output must equal, bit for bit, the device-pointer forward of the same
inputs (the kernels compute every image the same way whichever slice it is
in), and match the oracle."""
import numpy as np
import pytest

import synth
from parity_util import check_fp32, check_tf32, gpu_run, oracle_run

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
CASES = {
    "c2_tf32": (W["c2_min_tanh2"].resized(N=5, H=13), 0),                 # five slices of one image
    "c3_tf32": (W["c3_mul_lrelu_gelu"].resized(N=11, H=7), 0),            # eight slices of 1-2 images
    "c5_tf32": (W["c5_gn_pool_clamp"].resized(N=3, H=42), 0),             # GroupNorm, in-kernel finalize
    "c5_tf32_two_pass": (W["c5_gn_pool_clamp"].resized(N=5, H=12, W=140, Cout=128, groups=16), 0),  # conv, then post-pass
    "c5_tf32_half_bands": (W["c5_gn_pool_clamp"].resized(N=4, H=10, W=100, Cout=96, groups=12), 0),  # fused, 96 channels
    "c4_fp32": (W["c4_scale_min"].resized(N=4, H=7, W=96), 1),            # fp32 mode with channel indices
    "c2_fp32_odd": (W["c2_min_tanh2"].resized(N=3, H=9, W=31), 1),        # odd image sizes: one slice
    "c3_tf32_odd": (W["c3_mul_lrelu_gelu"].resized(N=3, H=6, W=37), 0),   # tf32 rows padded on the device
    # channels-last input (third field): in fp32 mode every slice transposes
    # its images into the handle's one NCHW copy, one slice after the other
    "c5_fp32_nhwc": (W["c5_gn_pool_clamp"].resized(N=5, H=14, W=36, Cin=6), 1, 1),
    "c2_fp32_nhwc": (W["c2_min_tanh2"].resized(N=9, H=8, W=40), 1, 1),
    "c4_tf32_nhwc": (W["c4_scale_min"].resized(N=3, H=7, W=64), 0, 1),
}


def host_run(wl, t, mode, want_index, layout=0):
    import x3_conv2d_epilogue_gb300 as ce
    chan = t.mult if wl.kind == synth.KIND_MUL_LRELU_GELU else t.scale
    probe = ce.epilogue(wl.kind, groups=wl.groups, pool_k=wl.pool_k, chan_scale=1, gamma=1, beta=1)
    shape = ce.conv_epi_output_shape(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, probe, mode)
    out = np.full(shape, np.nan, dtype=np.float32)
    idx = np.full(shape, -7, dtype=np.int32) if want_index else None
    epi = ce.epilogue(wl.kind, scalar=wl.scalar, chan_scale=chan, lrelu_slope=wl.lrelu_slope, groups=wl.groups,
                      eps=wl.eps, gamma=t.gamma, beta=t.beta, pool_k=wl.pool_k, clamp_lo=wl.clamp_lo,
                      clamp_hi=wl.clamp_hi, index_out=idx)
    h = ce.conv_epi_create(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, mode, layout)
    x = t.x.transpose(0, 2, 3, 1) if layout == ce.LAYOUT_NHWC else t.x
    try:
        ce.conv_epi_forward_host(h, np.ascontiguousarray(x), np.ascontiguousarray(t.w), np.ascontiguousarray(t.b),
                                 epi, out)
    finally:
        ce.conv_epi_destroy(h)
    return out, idx


@pytest.mark.parametrize("case", sorted(CASES))
def test_host_forward_matches_device_forward(case):
    import x3_conv2d_epilogue_gb300 as ce
    wl, fp32, *rest = CASES[case]
    layout = ce.LAYOUT_NHWC if rest and rest[0] else ce.LAYOUT_NCHW
    mode = ce.MODE_FP32 if fp32 else ce.MODE_TF32
    want_index = bool(fp32) and wl.kind != synth.KIND_MUL_LRELU_GELU
    t = synth.make_inputs(wl, seed=23)
    got, idx = host_run(wl, t, mode, want_index, layout)
    dev, dev_idx = gpu_run(wl, t, mode, want_index=want_index, layout=layout)
    np.testing.assert_array_equal(got, dev)
    if want_index:
        np.testing.assert_array_equal(idx, dev_idx)
    ref = oracle_run(wl, t)[0]
    (check_fp32 if fp32 else check_tf32)(got, ref, case + " host")
