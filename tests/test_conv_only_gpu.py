"""GPU parity of CONV_EPI_NONE, the conv output y itself with no chain, in
both arithmetic modes and both input layouts, against the oracle's direct
fp64 conv (every page's reference model: the nn.Conv2d layer whose output the
chain then consumes).

Small shapes run every tiling branch of the per-channel store path (row
tails, column tiles, channel tiles, padded rows, padded channels); the full
C3-sized problem is checked on sampled elements and on whole first and last
images' corner rows.  Integer inputs make the conv exact in both modes, and a
centre-tap filter turns it into the (rounded) input itself: both are bit
checks."""
import numpy as np
import pytest

import oracle
import synth
from parity_util import check_fp32, check_tf32, gpu_run, torch_inputs

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
NONE = synth.KIND_NONE
CASES = {
    "c3s": W["c3_mul_lrelu_gelu"].resized(N=2, H=11, kind=NONE),               # 9 rows: row pairs + a tail
    "c2s": W["c2_min_tanh2"].resized(N=2, H=21, kind=NONE),                    # Cin 16, Cout 64
    "c4s": W["c4_scale_min"].resized(N=1, H=12, kind=NONE),                    # Cout 128: one row per accumulator
    "c5s": W["c5_gn_pool_clamp"].resized(N=2, H=18, kind=NONE),                # Cin 8, 126-wide rows
    "w520": W["c3_mul_lrelu_gelu"].resized(N=1, H=5, W=520, kind=NONE),       # 3 column tiles
    "co200": W["c3_mul_lrelu_gelu"].resized(N=1, H=5, W=64, Cout=200, kind=NONE),  # 2 channel tiles, padded
    "co40": W["c3_mul_lrelu_gelu"].resized(N=1, H=9, W=128, Cout=40, kind=NONE),   # padded to 64 channels
    "w67": W["c3_mul_lrelu_gelu"].resized(N=2, H=6, W=67, kind=NONE),         # odd rows, padded input copy
    "w66": W["c3_mul_lrelu_gelu"].resized(N=1, H=7, W=66, kind=NONE),         # 64-wide rows: 16-byte aligned
    "w34": W["c3_mul_lrelu_gelu"].resized(N=1, H=7, W=34, Cin=4, kind=NONE),  # 32-wide rows, one chunk
    "cin3": W["c3_mul_lrelu_gelu"].resized(N=1, H=9, W=64, Cin=3, kind=NONE), # one zero-padded chunk
    "tiny": W["pr1_min_tanh2"].resized(N=1, Cin=1, H=3, W=4, Cout=1, kind=NONE),  # a 1 x 2 output
}


def modes():
    import x3_conv2d_epilogue_gb300 as ce
    return {"fp32": (ce.MODE_FP32, 0), "tf32": (ce.MODE_TF32, 0), "tf32_nhwc": (ce.MODE_TF32, ce.LAYOUT_NHWC)}


@pytest.mark.parametrize("mode", ["fp32", "tf32", "tf32_nhwc"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_conv_only_parity(case, mode):
    import x3_conv2d_epilogue_gb300 as ce
    wl = CASES[case]
    m, layout = modes()[mode]
    t = synth.make_inputs(wl, seed=4)
    if layout == ce.LAYOUT_NHWC and wl.Cin % 4 != 0:
        with pytest.raises(ce.ConvEpiError) as info:
            gpu_run(wl, t, m, layout=layout)
        assert ce.STATUS[info.value.status] == "UNSUPPORTED"
        return
    got, _ = gpu_run(wl, t, m, layout=layout)
    ref = oracle.conv3x3(t.x, t.w, t.b)
    assert got.shape == (wl.N, wl.Cout, wl.H - 2, wl.W - 2)
    (check_fp32 if mode == "fp32" else check_tf32)(got, ref, f"{case} {mode}")


@pytest.mark.parametrize("mode", ["fp32", "tf32"])
@pytest.mark.parametrize("case", ["c3s", "c4s", "w520", "co200"])
def test_conv_only_integer_inputs_bit_exact(case, mode):
    """Integer x, w, b with |v| <= 8: every product and partial sum is an
    integer below 2^24 and every operand fits tf32, so y is exact in both
    modes."""
    wl = CASES[case]
    t = synth.make_integer_inputs(wl, seed=6)
    got, _ = gpu_run(wl, t, modes()[mode][0])
    np.testing.assert_array_equal(got.astype(np.float64), oracle.conv3x3(t.x, t.w, t.b))


def tf32_rna(x: np.ndarray) -> np.ndarray:
    """fp32 -> tf32, 10 mantissa bits, round to nearest with ties away from zero."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x1000) & 0xFFFFE000).astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("mode", ["fp32", "tf32"])
def test_conv_only_centre_tap_reproduces_the_input(mode):
    """w[co, co % Cin, 1, 1] = 1, b = 0: y[n, co] is x[n, co % Cin] cropped by
    one pixel, exactly in fp32 mode and rounded to tf32 in tf32 mode (a single
    product by 1 and a single-term sum)."""
    wl = CASES["c3s"].resized(Cout=96)
    t = synth.make_inputs(wl, seed=8)
    t.w[:] = 0
    for co in range(wl.Cout):
        t.w[co, co % wl.Cin, 1, 1] = 1.0
    t.b[:] = 0
    got, _ = gpu_run(wl, t, modes()[mode][0])
    crop = t.x[:, np.arange(wl.Cout) % wl.Cin, 1:-1, 1:-1]
    want = crop if mode == "fp32" else tf32_rna(crop)
    np.testing.assert_array_equal(got.view(np.uint32), np.ascontiguousarray(want).view(np.uint32))


@pytest.mark.parametrize("mode", ["tf32", "fp32"])
def test_conv_only_full_size(mode):
    """The full C3-sized conv (x[64,64,256,256], 64 -> 64): 256 sampled
    elements (corners included) against the oracle's single-element conv, and
    the first and last output rows of every channel of the first and last
    images element by element."""
    import torch
    import x3_conv2d_epilogue_gb300 as ce
    wl = W["c3_mul_lrelu_gelu"].resized(kind=NONE)
    t = synth.make_inputs(wl, seed=0)
    d = torch_inputs(t)
    m = modes()[mode][0]
    epi = ce.epilogue(NONE)
    h = ce.conv_epi_create(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, m)
    try:
        out = torch.full(ce.conv_epi_output_shape(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, epi, m), float("nan"),
                         device="cuda", dtype=torch.float32)
        ce.conv_epi_forward(h, d["x"], d["w"], d["b"], epi, out)
        ce.conv_epi_sync(h)
    finally:
        ce.conv_epi_destroy(h)
    assert bool(torch.isfinite(out).all())
    tol = (lambda r: 1e-4) if mode == "fp32" else (lambda r: 5e-3 + 5e-3 * np.abs(r))
    rng = np.random.default_rng(77)
    Ho, Wo = wl.H - 2, wl.W - 2
    n, co = rng.integers(0, wl.N, 256), rng.integers(0, wl.Cout, 256)
    i, j = rng.integers(0, Ho, 256), rng.integers(0, Wo, 256)
    n[:2], co[:2], i[:2], j[:2] = [0, wl.N - 1], [0, wl.Cout - 1], [0, Ho - 1], [0, Wo - 1]
    ref = np.array([oracle.conv_at(t.x, t.w, t.b, int(a), int(c), int(p), int(q)) for a, c, p, q in zip(n, co, i, j)])
    got = out[torch.as_tensor(n), torch.as_tensor(co), torch.as_tensor(i), torch.as_tensor(j)].cpu().numpy()
    assert np.all(np.abs(got - ref) <= tol(ref))
    for img in (0, wl.N - 1):
        # rows 0..2 and Ho-3..Ho-1 of the image: a crop of the input that covers them
        for r0 in (0, Ho - 3):
            y = oracle.conv3x3(t.x[img:img + 1, :, r0:r0 + 5], t.w, t.b)[0]
            g = out[img, :, r0:r0 + 3].cpu().numpy().astype(np.float64)
            assert np.all(np.abs(g - y) <= tol(y)), (img, r0, float(np.abs(g - y).max()))
