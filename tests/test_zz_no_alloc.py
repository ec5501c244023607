"""The allocation-free forward (conv_epi_forward_noalloc) against the
ordinary handle-based forward and the oracle.

Some callers cannot allocate device memory: code running inside a custom
allocator or memory-pool callback, code that must not change the device's
memory footprint once it has started, or a runtime that lends the library
only its input and output buffers.  For them the library has one entry point
whose only scratch (the packed tf32 filter) is a fixed array in its own
device image.  It runs the same kernels as conv_epi_forward on the same
inputs, so its output must equal the handle forward's bit for bit, and stay
equal on a second call in a row although the array keeps the previous call's
contents (a call with another filter runs in between, so a stale packed
filter would show).  A call must not change the device's free memory, and a
barrier timeout on this path is reported by conv_epi_noalloc_sync, after
which the next call is correct again.  This file is collected last so a
failure here does not stop the rest of the suite from running.
"""
import numpy as np
import pytest

import synth
from parity_util import check_tf32, epilogue_for, gpu_run, oracle_run, torch_inputs

pytestmark = pytest.mark.gpu

CASES = {
    "c2_small": synth.WORKLOADS["c2_min_tanh2"].resized(N=2, H=21),
    "c4_small": synth.WORKLOADS["c4_scale_min"].resized(N=1, H=12),
    "c3_small": synth.WORKLOADS["c3_mul_lrelu_gelu"].resized(N=2, H=11),
    "conv_only": synth.WORKLOADS["c3_mul_lrelu_gelu"].resized(N=2, H=11, kind=synth.KIND_NONE),
}


def noalloc(wl, d, epi, out):
    import x3_conv2d_epilogue_gb300 as ce
    ce.conv_epi_forward_noalloc(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, d["x"], d["w"], d["b"], epi, out)


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_handle_forward_twice(case):
    import torch
    import x3_conv2d_epilogue_gb300 as ce
    wl = CASES[case]
    t = synth.make_inputs(wl, seed=11)
    ref, _ = gpu_run(wl, t, ce.MODE_TF32)            # handle-based entry point
    want = oracle_run(wl, t)[0] if wl.kind != synth.KIND_NONE else None
    d = torch_inputs(t)
    epi = epilogue_for(wl, d)
    other = torch_inputs(synth.make_inputs(wl, seed=12))   # another filter for the call in between
    other_out = torch.empty(ref.shape, device="cuda", dtype=torch.float32)
    out = torch.empty(ref.shape, device="cuda", dtype=torch.float32)
    for call in range(2):
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        noalloc(wl, d, epi, out)
        ce.conv_epi_noalloc_sync()
        free1, alloc1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        got = out.cpu().numpy()
        np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32), err_msg=f"call {call}")
        if want is not None:
            check_tf32(got, want, f"{case} call {call}")
        if call == 1:   # the call's kernels are loaded by now: nothing may change the footprint
            assert (free1, alloc1) == (free0, alloc0), f"device memory changed: {free0 - free1} bytes"
        # the array now holds another filter's packed copy
        noalloc(wl, other, epilogue_for(wl, other), other_out)
        ce.conv_epi_noalloc_sync()


def test_noalloc_timeout_is_reported_and_the_next_call_recovers():
    """conv_epi_test_drop_tile(None, 0) makes the next allocation-free
    forward's producers skip their first staged tile, so the converters'
    bounded waits run out (about 2 s, no fault); conv_epi_noalloc_sync
    reports the timeout once and clears it, and the next call equals the
    handle forward again."""
    import time

    import torch
    import x3_conv2d_epilogue_gb300 as ce
    wl = CASES["c4_small"]
    t = synth.make_inputs(wl, seed=13)
    ref, _ = gpu_run(wl, t, ce.MODE_TF32)
    d = torch_inputs(t)
    epi = epilogue_for(wl, d)
    out = torch.empty(ref.shape, device="cuda", dtype=torch.float32)
    ce.conv_epi_noalloc_sync()                       # nothing pending
    ce.conv_epi_test_drop_tile(None, 0)
    t0 = time.perf_counter()
    noalloc(wl, d, epi, out)
    with pytest.raises(ce.ConvEpiError) as info:
        ce.conv_epi_noalloc_sync()
    assert ce.STATUS[info.value.status] == "TIMEOUT"
    assert 1.5 < time.perf_counter() - t0 < 30
    ce.conv_epi_noalloc_sync()                       # cleared
    out.fill_(float("nan"))
    noalloc(wl, d, epi, out)
    ce.conv_epi_noalloc_sync()
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


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
    # the same statuses as the handle forward for a bad chain description
    idx = torch.zeros(1, 64, 6, 6, device="cuda", dtype=torch.int32)
    o3 = torch.zeros(1, 64, 6, 6, device="cuda")
    bad = ce.epilogue(ce.MUL_LRELU_GELU, chan_scale=p, index_out=idx)
    with pytest.raises(ce.ConvEpiError) as ei:
        ce.conv_epi_forward_noalloc(1, 8, 8, 8, 64, x, w, b, bad, o3)
    h = ce.conv_epi_create(1, 8, 8, 8, 64)
    try:
        with pytest.raises(ce.ConvEpiError) as eh:
            ce.conv_epi_forward(h, x, w, b, bad, o3)
    finally:
        ce.conv_epi_destroy(h)
    assert ei.value.status == eh.value.status == 1
