"""conv_epi_postpass: each chain as a separate pass over a stored conv output
(the unfused design the pages plan their kernels for), against the oracle's
chain on the same float32 conv output, element by element within the fp32
bound (1e-4); and cuDNN's conv (PyTorch, fp32) followed by the pass against
the oracle's whole forward, which is what the bench's unfused comparator
computes."""
import numpy as np
import pytest

import oracle
import synth
from parity_util import FP32_ATOL, check_fp32, epilogue_for, torch_inputs

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
CASES = {
    "pr1": W["pr1_min_tanh2"],
    "c2s": W["c2_min_tanh2"].resized(N=2, H=21),
    "c4s": W["c4_scale_min"].resized(N=1, H=12),
    "c4neg": W["c4_scale_min"].resized(N=1, H=7, W=96, scalar=-1.5),
    "c4_co200": W["c4_scale_min"].resized(N=1, H=6, W=64, Cout=200),
    "c3s": W["c3_mul_lrelu_gelu"].resized(N=2, H=11),
    "c3_w67": W["c3_mul_lrelu_gelu"].resized(N=2, H=6, W=67),          # 4 x 65 = 260-float planes: 16-byte path
    "c3_p325": W["c3_mul_lrelu_gelu"].resized(N=1, H=7, W=67, Cin=5),  # 5 x 65 = 325-float planes: one float per thread
    "none": W["c3_mul_lrelu_gelu"].resized(N=2, H=9, kind=synth.KIND_NONE),
    "c5s": W["c5_gn_pool_clamp"].resized(N=2, H=42),
    "c5g1": W["c5_gn_pool_clamp"].resized(N=1, H=22, groups=1),
    "c5g4": W["c5_gn_pool_clamp"].resized(N=1, H=18, groups=4),
    "c5_w37": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=37),
    "c5_k2": W["c5_gn_pool_clamp"].resized(N=1, H=14, W=30, pool_k=2),
    "c5_co32": W["c5_gn_pool_clamp"].resized(N=2, H=14, W=40, Cout=32, groups=8),
    # each instantiation of the pooling pass: 4 x 4 windows by 16-byte loads
    # (Wo a multiple of 4), 2 x 2 by single floats (odd Wo), no pooling, 3 x 3,
    # and a window size taken at run time
    "c5_k4_v4": W["c5_gn_pool_clamp"].resized(N=1, H=13, W=34),
    "c5_k2_odd": W["c5_gn_pool_clamp"].resized(N=1, H=12, W=31, pool_k=2),
    "c5_k1": W["c5_gn_pool_clamp"].resized(N=1, H=9, W=20, pool_k=1, groups=4),
    "c5_k3": W["c5_gn_pool_clamp"].resized(N=1, H=14, W=29, pool_k=3),
    "c5_k5": W["c5_gn_pool_clamp"].resized(N=1, H=17, W=27, pool_k=5),
}


def oracle_chain(wl, t, y):
    if wl.kind == synth.KIND_NONE:
        return y
    if wl.kind in (synth.KIND_MIN_TANH2, synth.KIND_SCALE_MIN):
        return oracle.chain_min(y, wl.scalar, wl.kind == synth.KIND_MIN_TANH2)[0]
    if wl.kind == synth.KIND_MUL_LRELU_GELU:
        return oracle.chain_mul_lrelu_gelu(y, t.mult, wl.lrelu_slope)
    return oracle.chain_gn_pool(y, oracle.chain_for(wl, t))[0]


def postpass(wl, d, y_dev):
    import torch
    import x3_conv2d_epilogue_gb300 as ce
    epi = epilogue_for(wl, d)
    h = ce.conv_epi_create(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, ce.MODE_FP32)
    try:
        out = torch.full(ce.conv_epi_output_shape(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, epi, ce.MODE_FP32), float("nan"),
                         device="cuda", dtype=torch.float32)
        ce.conv_epi_postpass(h, y_dev, epi, out)
        ce.conv_epi_sync(h)
    finally:
        ce.conv_epi_destroy(h)
    return out.cpu().numpy()


@pytest.mark.parametrize("case", sorted(CASES))
def test_postpass_matches_the_oracle_chain(case):
    import torch
    wl = CASES[case]
    t = synth.make_inputs(wl, seed=21)
    y32 = oracle.conv3x3(t.x, t.w, t.b).astype(np.float32)
    got = postpass(wl, torch_inputs(t), torch.from_numpy(y32).cuda())
    check_fp32(got, oracle_chain(wl, t, y32.astype(np.float64)), case)


@pytest.mark.parametrize("case", ["c2s", "c3s", "c4neg", "c5s"])
def test_cudnn_conv_then_postpass_matches_the_oracle(case):
    """The bench's unfused comparator in fp32: cuDNN's conv writes y in full,
    then the one post-pass."""
    import torch
    import torch.nn.functional as F
    wl = CASES[case]
    t = synth.make_inputs(wl, seed=22)
    d = torch_inputs(t)
    torch.backends.cudnn.allow_tf32 = False
    y = F.conv2d(d["x"], d["w"], d["b"]).contiguous()
    got = postpass(wl, d, y)
    ref = oracle.forward(t.x, t.w, t.b, oracle.chain_for(wl, t))[0]
    err = np.abs(got.astype(np.float64) - ref)
    assert err.max() <= 2 * FP32_ATOL, f"{case}: max err {err.max():.3g}"


def test_postpass_arguments():
    import torch
    import x3_conv2d_epilogue_gb300 as ce
    h = ce.conv_epi_create(1, 8, 10, 12, 64, ce.MODE_FP32)
    try:
        y = torch.zeros(1, 64, 8, 10, device="cuda")
        out = torch.zeros(1, 1, 8, 10, device="cuda")
        idx = torch.zeros(1, 1, 8, 10, device="cuda", dtype=torch.int32)
        with pytest.raises(ce.ConvEpiError) as ei:
            ce.conv_epi_postpass(h, y, ce.epilogue(ce.SCALE_MIN, index_out=idx), out)
        assert ce.STATUS[ei.value.status] == "UNSUPPORTED"
        flat = torch.zeros(64 * 80 + 4, device="cuda")
        with pytest.raises(ce.ConvEpiError) as ei:      # y not 16-byte aligned
            ce.conv_epi_postpass(h, flat[1:].data_ptr(), ce.epilogue(ce.SCALE_MIN), out)
        assert ce.STATUS[ei.value.status] == "ALIGNMENT"
        ce.conv_epi_postpass(h, y, ce.epilogue(ce.SCALE_MIN, scalar=2.0), out)
        ce.conv_epi_sync(h)
        assert float(out.abs().max()) == 0.0
    finally:
        ce.conv_epi_destroy(h)
    h0 = ce.conv_epi_create(0, 8, 10, 12, 64, ce.MODE_FP32)   # an empty batch: nothing to do
    try:
        ce.conv_epi_postpass(h0, 0, ce.epilogue(ce.MIN_TANH2), 0)
    finally:
        ce.conv_epi_destroy(h0)
