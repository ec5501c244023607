"""Failure detection on the GPU without a fault: every barrier wait of the
tensor-core kernel is bounded.  The library's test hook makes one staged
input tile per CTA never arrive (its copy is neither issued nor announced),
so the waits on that slot run out.  The forward must report
CONV_EPI_ERR_TIMEOUT through conv_epi_sync(), after roughly the wait limit,
and the same handle must then run a normal forward to full parity: the
context survived and the hook applied to one forward only.

Nothing here traps, faults or hangs the GPU: the abandoned slot has no copy
in flight, every other copy and MMA is drained before the CTA exits, and
each wait gives up after 2 s.
"""
import time

import numpy as np
import pytest

import synth
from parity_util import check_tf32, epilogue_for, oracle_run, torch_inputs

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
CASES = {
    # filter resident in shared memory; the producer blocks on the tile ring
    "c2_resident": (W["c2_min_tanh2"].resized(N=2, H=21), 1, 0),
    # filter streamed (Cin 64): the producer polls both rings without blocking
    "c3_streamed": (W["c3_mul_lrelu_gelu"].resized(N=2, H=11), 2, 0),
    # GroupNorm chain: the finalize kernel still runs after the timed-out conv
    "c5_gn_first_tile": (W["c5_gn_pool_clamp"].resized(N=2, H=42), 0, 0),
    # channels-last input: the dropped copy is a B plane, so the MMA thread's
    # wait is the one that runs out
    "c4_channels_last": (W["c4_scale_min"].resized(N=1, H=12), 3, 1),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_dropped_tile_times_out_then_recovers(case):
    import torch
    import x3_conv2d_epilogue_gb300 as ce
    wl, tile, layout = CASES[case]
    t = synth.make_inputs(wl, seed=21)
    d = torch_inputs(t)
    if layout == ce.LAYOUT_NHWC:
        d["x"] = d["x"].permute(0, 2, 3, 1).contiguous()
    probe = ce.epilogue(wl.kind, groups=wl.groups, pool_k=wl.pool_k, chan_scale=1, gamma=1, beta=1)
    shape = ce.conv_epi_output_shape(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, probe, ce.MODE_TF32)
    out = torch.full(shape, float("nan"), device="cuda", dtype=torch.float32)
    epi = epilogue_for(wl, d)
    h = ce.conv_epi_create(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, ce.MODE_TF32, layout)
    try:
        ce.conv_epi_test_drop_tile(h, tile)
        t0 = time.perf_counter()
        ce.conv_epi_forward(h, d["x"], d["w"], d["b"], epi, out)
        with pytest.raises(ce.ConvEpiError) as info:
            ce.conv_epi_sync(h)
        elapsed = time.perf_counter() - t0
        assert ce.STATUS[info.value.status] == "TIMEOUT", str(info.value)
        # the converters give up after the 2 s limit; the other roles follow
        # the abort flag, so the whole kernel ends soon after
        assert 1.5 < elapsed < 30.0, elapsed
        # the error word was cleared by the sync that reported it
        ce.conv_epi_sync(h)
        # same handle, hook consumed: a normal forward matches the oracle
        out.fill_(float("nan"))
        ce.conv_epi_forward(h, d["x"], d["w"], d["b"], epi, out)
        ce.conv_epi_sync(h)
    finally:
        ce.conv_epi_destroy(h)
    torch.cuda.synchronize()
    check_tf32(out.cpu().numpy(), oracle_run(wl, t)[0], case)


def test_drop_tile_hook_arguments():
    import x3_conv2d_epilogue_gb300 as ce
    wl = W["pr1_min_tanh2"]
    h = ce.conv_epi_create(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, ce.MODE_FP32)
    try:
        with pytest.raises(ce.ConvEpiError) as info:
            ce.conv_epi_test_drop_tile(h, 0)  # the fp32 kernels have no barrier rings
        assert ce.STATUS[info.value.status] == "UNSUPPORTED"
    finally:
        ce.conv_epi_destroy(h)
    h = ce.conv_epi_create(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, ce.MODE_TF32)
    try:
        with pytest.raises(ce.ConvEpiError):
            ce.conv_epi_test_drop_tile(h, -2)
        ce.conv_epi_test_drop_tile(h, 3)
        ce.conv_epi_test_drop_tile(h, -1)  # cancelled: the next forward is normal
        t = synth.make_inputs(wl, seed=4)
        d = torch_inputs(t)
        import torch
        out = torch.full((wl.N, 1, wl.H - 2, wl.W - 2), float("nan"), device="cuda", dtype=torch.float32)
        ce.conv_epi_forward(h, d["x"], d["w"], d["b"], epilogue_for(wl, d), out)
        ce.conv_epi_sync(h)
    finally:
        ce.conv_epi_destroy(h)
    check_tf32(out.cpu().numpy(), oracle_run(wl, t)[0], "cancelled hook")
