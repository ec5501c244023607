"""Debug handles (CONV_EPI_DEBUG=1 when the handle is created): the forward
waits for its own stream, so a device-side barrier timeout is returned by
conv_epi_forward itself rather than by a later conv_epi_sync.  The timeout
is made with the library's drop-a-copy test hook (no fault, no hang: the
waits give up after their 2 s limit).  Collected near the end of the suite.
"""
import pytest

import synth
from parity_util import check_tf32, epilogue_for, oracle_run, torch_inputs

pytestmark = pytest.mark.gpu


def test_debug_forward_returns_the_timeout(monkeypatch):
    import torch
    import x3_conv2d_epilogue_gb300 as ce
    wl = synth.WORKLOADS["c2_min_tanh2"].resized(N=2, H=21)
    t = synth.make_inputs(wl, seed=23)
    d = torch_inputs(t)
    epi = epilogue_for(wl, d)
    out = torch.full((wl.N, 1, wl.H - 2, wl.W - 2), float("nan"), device="cuda")
    monkeypatch.setenv("CONV_EPI_DEBUG", "1")
    h = ce.conv_epi_create(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, ce.MODE_TF32)
    monkeypatch.delenv("CONV_EPI_DEBUG")
    try:
        ce.conv_epi_test_drop_tile(h, 1)
        with pytest.raises(ce.ConvEpiError) as info:
            ce.conv_epi_forward(h, d["x"], d["w"], d["b"], epi, out)
        assert ce.STATUS[info.value.status] == "TIMEOUT"
        ce.conv_epi_sync(h)                      # the error word was already cleared
        out.fill_(float("nan"))
        ce.conv_epi_forward(h, d["x"], d["w"], d["b"], epi, out)   # returns OK after its own sync
    finally:
        ce.conv_epi_destroy(h)
    check_tf32(out.cpu().numpy(), oracle_run(wl, t)[0], "debug handle")

