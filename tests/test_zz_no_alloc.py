"""The allocation-free forward (conv_epi_forward_noalloc) against the
ordinary handle-based forward.

Some callers cannot allocate device memory (allocator or memory-pool
callbacks, runtimes that only lend the library its input and output
buffers), so the library offers one entry point whose scratch is a fixed
array in its own device image.  It must give the same result as
conv_epi_forward on the same inputs, and keep doing so on a second call in a
row (the array keeps the previous call's contents).  This file is collected
last so a failure here does not stop the rest of the suite from running.
"""
import numpy as np
import pytest

import synth
from parity_util import TF32_ATOL, TF32_RTOL, epilogue_for, gpu_run, torch_inputs

pytestmark = pytest.mark.gpu

CASES = {
    "c2_small": synth.WORKLOADS["c2_min_tanh2"].resized(N=2, H=21),
    "c4_small": synth.WORKLOADS["c4_scale_min"].resized(N=1, H=12),
    "c3_small": synth.WORKLOADS["c3_mul_lrelu_gelu"].resized(N=2, H=11),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_handle_forward_twice(case):
    import torch
    import x3_conv2d_epilogue_gb300 as ce
    wl = CASES[case]
    t = synth.make_inputs(wl, seed=11)
    ref, _ = gpu_run(wl, t, ce.MODE_TF32)            # handle-based entry point
    d = torch_inputs(t)
    epi = epilogue_for(wl, d)
    for call in range(2):                             # the array keeps the previous call's contents
        out = torch.full(ref.shape, float("nan"), device="cuda", dtype=torch.float32)
        ce.conv_epi_forward_noalloc(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, d["x"], d["w"], d["b"], epi, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        err = np.abs(got.astype(np.float64) - ref)
        assert np.all(np.isfinite(got)), f"call {call}: non-finite output"
        assert np.all(err <= TF32_ATOL + TF32_RTOL * np.abs(ref)), f"call {call}: max diff {err.max():.3g}"


def test_noalloc_refuses_what_it_cannot_hold():
    import torch
    import x3_conv2d_epilogue_gb300 as ce
    x = torch.zeros(1, 8, 8, 8, device="cuda")
    w = torch.zeros(64, 8, 3, 3, device="cuda")
    b = torch.zeros(64, device="cuda")
    p = torch.ones(64, device="cuda")
    out = torch.zeros(1, 64, 1, 1, device="cuda")
    gn = ce.epilogue(ce.GN_SCALE_POOL_CLAMP, chan_scale=p, gamma=p, beta=b, groups=16, pool_k=4)
    with pytest.raises(ce.ConvEpiError) as ei:        # GroupNorm chain needs a workspace
        ce.conv_epi_forward_noalloc(1, 8, 8, 8, 64, x, w, b, gn, out)
    assert ei.value.status == 2
    big_w = torch.zeros(128, 512, 3, 3, device="cuda")   # packed filter larger than the array
    xb = torch.zeros(1, 512, 8, 8, device="cuda")
    ob = torch.zeros(1, 1, 6, 6, device="cuda")
    with pytest.raises(ce.ConvEpiError) as ei:
        ce.conv_epi_forward_noalloc(1, 512, 8, 8, 128, xb, big_w, p.repeat(2), ce.epilogue(ce.SCALE_MIN), ob)
    assert ei.value.status == 2
    xo = torch.zeros(1, 8, 8, 7, device="cuda")            # NCHW rows of 7 floats need the padded copy
    oo = torch.zeros(1, 1, 6, 5, device="cuda")
    with pytest.raises(ce.ConvEpiError) as ei:
        ce.conv_epi_forward_noalloc(1, 8, 8, 7, 64, xo, w, b, ce.epilogue(ce.SCALE_MIN), oo)
    assert ei.value.status == 2
