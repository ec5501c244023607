"""The forward inside a CUDA graph: after conv_epi_reserve (so the forward
allocates nothing), a conv_epi_forward captured on a stream and replayed
gives the same outputs as a direct call, for a min chain, the per-channel
chain and the GroupNorm chain (whose fused tf32 form is a cooperative launch
plus a memset of its arrival counter, and whose two-pass form is the conv
and the post-pass's kernels), and for rows that the library first copies
into 16-byte-padded rows."""
import numpy as np
import pytest

import synth
from parity_util import check_tf32, epilogue_for, oracle_run, torch_inputs

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
CASES = {
    "c2": W["c2_min_tanh2"].resized(N=2, H=21),
    "c3": W["c3_mul_lrelu_gelu"].resized(N=1, H=9),
    "c5": W["c5_gn_pool_clamp"].resized(N=2, H=42),
    "c2_w63": W["c2_min_tanh2"].resized(N=2, H=9, W=63),    # the row-padding kernel is captured too
    # GroupNorm in two passes (conv into the handle's buffer, then the
    # post-pass): both buffers come from conv_epi_reserve
    "c5_two_pass": W["c5_gn_pool_clamp"].resized(N=2, H=14, W=150, Cout=128, groups=16, pool_k=2),
    # GroupNorm over 128 channels fused in half bands (the generalised instantiation)
    "c5_half_bands": W["c5_gn_pool_clamp"].resized(N=2, H=14, W=110, Cout=128, groups=16),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_forward_replays_in_a_cuda_graph(case):
    import torch
    import x3_conv2d_epilogue_gb300 as ce
    wl = CASES[case]
    t = synth.make_inputs(wl, seed=17)
    d = torch_inputs(t)
    epi = epilogue_for(wl, d)
    h = ce.conv_epi_create(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, ce.MODE_TF32)
    try:
        ce.conv_epi_reserve(h, epi)
        shape = ce.conv_epi_output_shape(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, epi)
        direct = torch.full(shape, float("nan"), device="cuda")
        ce.conv_epi_forward(h, d["x"], d["w"], d["b"], epi, direct)
        ce.conv_epi_sync(h)
        out = torch.full(shape, float("nan"), device="cuda")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            ce.conv_epi_forward(h, d["x"], d["w"], d["b"], epi, out, s)
        for _ in range(3):
            out.fill_(float("nan"))
            g.replay()
        torch.cuda.synchronize()
        ce.conv_epi_sync(h)
    finally:
        ce.conv_epi_destroy(h)
    got = out.cpu().numpy()
    np.testing.assert_array_equal(got, direct.cpu().numpy())
    check_tf32(got, oracle_run(wl, t)[0], case + " graph")
