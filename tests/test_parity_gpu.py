"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, on
the same seeded inputs, element by element.

Small cases keep every workload's chain, channel counts and filter size but
shrink N and H (and sometimes W) so the oracle finishes in seconds while the
kernels still run several tiles and a ragged tail.
"""
import numpy as np
import pytest

import oracle
import synth
from parity_util import (check_fp32, check_index, check_tf32, fp32_indices, gpu_run, min_index_gap, oracle_run,
                         pool_index_gap)

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
SMALL = {
    "pr1": W["pr1_min_tanh2"],
    "c2s": W["c2_min_tanh2"].resized(N=2, H=21),                              # 19 output rows (odd tail)
    "c2w": W["c2_min_tanh2"].resized(N=1, H=9, W=200),                        # ragged row width
    "c3s": W["c3_mul_lrelu_gelu"].resized(N=2, H=11),
    "c4s": W["c4_scale_min"].resized(N=1, H=12),
    "c4neg": W["c4_scale_min"].resized(N=1, H=7, W=96, scalar=-1.5),          # max branch
    "c5s": W["c5_gn_pool_clamp"].resized(N=2, H=42),                         # 40 rows: 10 bands, no tail
    "c5t": W["c5_gn_pool_clamp"].resized(N=2, H=40),                         # 38 rows: 9 bands + 2 stat rows
    "c4w128": W["c4_scale_min"].resized(N=1, H=9, W=128),                    # tf32 converter falls back to single items
    "c2w64": W["c2_min_tanh2"].resized(N=2, H=23, W=64),                     # four row pairs per accumulator, ragged units
    "c2cin12": W["c2_min_tanh2"].resized(N=1, H=11, Cin=12),                 # Cin not a multiple of 8 (zero-padded chunk)
    "c3cin3": W["c3_mul_lrelu_gelu"].resized(N=1, H=9, W=64, Cin=3),        # 3 input channels (one padded chunk)
    "c4cin20": W["c4_scale_min"].resized(N=1, H=7, Cin=20),                  # Cout 128, Cin 20
    "c2co48": W["c2_min_tanh2"].resized(N=1, H=9, Cout=48),                  # Cout padded to 64 (zero filters)
    "c4co100": W["c4_scale_min"].resized(N=1, H=7, W=128, Cout=100, scalar=-0.5),  # padded to 128, max branch
    "c3co40": W["c3_mul_lrelu_gelu"].resized(N=1, H=9, W=128, Cout=40),      # per-channel stores skip padding
    "c5g1": W["c5_gn_pool_clamp"].resized(N=1, H=22, groups=1),               # one group: 64 channels over two quadrants
    "c5g4": W["c5_gn_pool_clamp"].resized(N=1, H=18, groups=4),               # 16 channels per group
    # degenerate and boundary shapes
    "min_cout1": W["pr1_min_tanh2"].resized(N=1, Cin=1, H=3, W=4, Cout=1),   # one input and one output channel, 1 x 2 output
    "c2_w4": W["c2_min_tanh2"].resized(N=1, H=8, W=4),                       # two output columns
    "c4_one_row": W["c4_scale_min"].resized(N=2, H=3, W=64),                 # one output row per image
    "c2_cin256": W["c2_min_tanh2"].resized(N=1, H=6, W=64, Cin=256),          # 32 input chunks, filter streamed
    "c3_cout1": W["c3_mul_lrelu_gelu"].resized(N=1, H=5, W=32, Cout=1),      # a single per-channel row
    "c5_w16": W["c5_gn_pool_clamp"].resized(N=2, H=10, W=16),                # 3 pooled columns, 2 pooled rows (two bands per unit)
    "c5_w64": W["c5_gn_pool_clamp"].resized(N=2, H=22, W=64),                # two bands per unit, the last unit's second band past Hp
    "c5_w40": W["c5_gn_pool_clamp"].resized(N=1, H=14, W=40, groups=4),      # rows padded to 64 columns
    "c5_one_band": W["c5_gn_pool_clamp"].resized(N=1, H=6),                  # one pooling band per image
    # rows wider than one tile (the tf32 path splits them into column tiles of 252 outputs)
    "c2_w300": W["c2_min_tanh2"].resized(N=1, H=6, W=300),                   # 2 tiles: 252 + 46 columns
    "c3_w520": W["c3_mul_lrelu_gelu"].resized(N=1, H=5, W=520),              # 3 tiles, per-channel stores
    "c4_w516": W["c4_scale_min"].resized(N=2, H=4, W=516, scalar=-1.0),      # 3 tiles, Cout 128, max branch
    "c5_w260": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=260),              # GroupNorm over 2 column tiles, the last 6 columns
    "c5_w200": W["c5_gn_pool_clamp"].resized(N=2, H=15, W=200),              # wide rows: 49 windows, half bands, a stats-only row
    "c5_w256": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=256, groups=4),    # wide rows, P 256: 63 windows
    "c5_w130": W["c5_gn_pool_clamp"].resized(N=1, H=9, W=130, Cout=32, groups=8),  # Wo 128, 32 channels
    "c5_w129": W["c5_gn_pool_clamp"].resized(N=1, H=9, W=129),              # Wo 127: one column tile, its first pass masked
    # more than 128 output channels (the tf32 path runs channel tiles of 128)
    "c4_co256": W["c4_scale_min"].resized(N=1, H=5, W=64, Cout=256),        # 2 channel tiles, atomic minimum
    "c3_co200": W["c3_mul_lrelu_gelu"].resized(N=1, H=5, W=64, Cout=200),   # 2 tiles, the second padded
    "c2_co300_w300": W["c2_min_tanh2"].resized(N=1, H=4, W=300, Cout=300),  # 3 channel x 2 column tiles
    # rows whose width is not a multiple of 4 (the tf32 path copies NCHW input
    # into rows padded to whole 16-byte units first; channels last needs no copy)
    "c2_w255": W["c2_min_tanh2"].resized(N=1, H=7, W=255),                   # 253 outputs per row
    "c3_w67": W["c3_mul_lrelu_gelu"].resized(N=2, H=6, W=67),               # odd output rows: scalar stores
    "c4_w262": W["c4_scale_min"].resized(N=1, H=4, W=262),                   # 2 column tiles over padded rows
    "c5_w126": W["c5_gn_pool_clamp"].resized(N=1, H=18, W=126),              # 124 columns: 31 whole windows
    "c5_w37": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=37),                # two bands per unit, 3 columns past the pool
    "c5_w98": W["c5_gn_pool_clamp"].resized(N=1, H=14, W=98),                # fused, 112 columns: chunk 6 whole, chunk 7 absent
    "c5_w107": W["c5_gn_pool_clamp"].resized(N=1, H=13, W=107),              # fused, chunk 6 ragged at column 105
    "c5_w90": W["c5_gn_pool_clamp"].resized(N=1, H=12, W=90),                # one band of 96 columns (generalised kernel)
    "c5_w66": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=66),                # Wo 64 in P 80: chunk 4 all masked
    "c5_w65": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=65),                # Wo 63: two passes in tf32
    "c5_co128_w80": W["c5_gn_pool_clamp"].resized(N=1, H=11, W=80, Cout=128, groups=32),  # half bands in P 80
    "min_w3": W["pr1_min_tanh2"].resized(N=2, Cin=2, H=3, W=3, Cout=1),      # a single output per image
    # GroupNorm shapes beyond the page's (tf32: fused where the epilogue takes
    # them, else the conv then the chain's post-pass through a buffer of y)
    "c5_co32": W["c5_gn_pool_clamp"].resized(N=2, H=18, W=64, Cout=32, groups=8),     # Cout 32 (fused: 32 zero filters)
    "c5_co16_w128": W["c5_gn_pool_clamp"].resized(N=1, H=14, W=128, Cout=16, groups=2),  # Cout 16, one band, 8 per group
    "c5_co48": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=64, Cout=48, groups=16),    # 3 channels per group: two passes
    "c5_co128": W["c5_gn_pool_clamp"].resized(N=1, H=14, W=96, Cout=128, groups=16),  # Cout 128, W 96: half bands, P 96
    "c5_co128_w128": W["c5_gn_pool_clamp"].resized(N=2, H=15, W=128, Cout=128, groups=16),  # fused, half bands, a stats-only row
    "c5_co96_w100": W["c5_gn_pool_clamp"].resized(N=1, H=14, W=100, Cout=96, groups=12),  # fused, 32 zero filters, P 112
    "c5_co128_g2": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=110, Cout=128, groups=2),   # fused, 64 channels per group
    "c5_co256": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=64, Cout=256, groups=32),  # 2 channel tiles, W 64: whole bands per tile
    "c5_k2": W["c5_gn_pool_clamp"].resized(N=2, H=13, W=50, pool_k=2),               # 2 x 2 windows, odd tail row (four bands per unit)
    "c5_k2_w64": W["c5_gn_pool_clamp"].resized(N=1, H=19, W=64, Cout=32, groups=8, pool_k=2),  # a unit of one valid row
    "c5_k2_w20": W["c5_gn_pool_clamp"].resized(N=2, H=12, W=20, pool_k=2, groups=4),          # 9 windows
    "c5_k2_co128_w64": W["c5_gn_pool_clamp"].resized(N=2, H=11, W=64, Cout=128, groups=16, pool_k=2),  # no stacking, two bands per unit
    "c5_k2_co80_w30": W["c5_gn_pool_clamp"].resized(N=1, H=14, W=30, Cout=80, groups=5, pool_k=2),     # 48 zero filters, 16 per group
    "c5_k2_w200": W["c5_gn_pool_clamp"].resized(N=1, H=11, W=200, pool_k=2),                  # rows of 198 outputs, 99 windows
    "c5_k2_w240": W["c5_gn_pool_clamp"].resized(N=2, H=8, W=240, Cout=32, groups=8, pool_k=2),  # 119 windows
    "c5_k2_w256": W["c5_gn_pool_clamp"].resized(N=1, H=8, W=256, Cout=32, groups=8, pool_k=2),  # NCHW two passes; channels last fused, 127 windows
    "c5_k1": W["c5_gn_pool_clamp"].resized(N=1, H=9, W=33, pool_k=1, groups=4),      # no pooling
    # fp32 GroupNorm staging: two input-channel steps (rows staged per output
    # row), and bands staged at once with rows of odd width and a short last band
    "c5_cin20": W["c5_gn_pool_clamp"].resized(N=1, H=15, W=40, Cin=20),
    "c5_cin13_w37": W["c5_gn_pool_clamp"].resized(N=2, H=12, W=37, Cin=13, Cout=32, groups=8),
    "c5_cin16_k2": W["c5_gn_pool_clamp"].resized(N=1, H=11, W=52, Cin=16, pool_k=2),
    "c5_k2_w300": W["c5_gn_pool_clamp"].resized(N=1, H=8, W=300, pool_k=2, groups=64),  # 2 column tiles, a group per channel
    # GroupNorm shapes the fp32 kernel does not take (two passes there, no indices; tf32 too for pool_k 3)
    "c5_k3": W["c5_gn_pool_clamp"].resized(N=1, H=14, W=29, pool_k=3),
    "c5_co128_g128": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=100, Cout=128, groups=128),  # 128 groups
    # 2 x 2 windows fused (Cout <= 64, W 66..128: two bands of 2 rows per unit)
    "c5_k2_w128": W["c5_gn_pool_clamp"].resized(N=2, H=13, W=128, pool_k=2),        # 63 windows, a stats-only tail row
    "c5_k2_w90": W["c5_gn_pool_clamp"].resized(N=1, H=12, W=90, Cout=32, groups=8, pool_k=2),  # P 96, masked chunks
    "c5_k2_w67": W["c5_gn_pool_clamp"].resized(N=1, H=15, W=67, pool_k=2, groups=1),  # odd Wo: a stats-only column; one group
    "c5_k2_w66": W["c5_gn_pool_clamp"].resized(N=2, H=9, W=66, Cout=48, groups=12, pool_k=2),  # Wo 64, 48 channels
    "c5_k2_g64": W["c5_gn_pool_clamp"].resized(N=2, H=12, W=100, groups=64, pool_k=2),  # a group per channel: 245-float blocks, separate finalize
    "c5_k2_co128": W["c5_gn_pool_clamp"].resized(N=2, H=13, W=100, Cout=128, groups=16, pool_k=2),  # no stacking, a stats-only row
    "c5_k2_co96_w128": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=128, Cout=96, groups=12, pool_k=2),  # 32 zero filters, 63 windows
    # 65..128 channels in rows of up to 64 columns: no stacking, one whole band per unit
    "c5_co128_w64": W["c5_gn_pool_clamp"].resized(N=2, H=13, W=64, Cout=128, groups=16),  # a stats-only unit
    "c5_co96_w40": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=40, Cout=96, groups=12),   # 32 zero filters, 9 windows
    "c5_co320_w50": W["c5_gn_pool_clamp"].resized(N=2, H=11, W=50, Cout=320, groups=10),  # 3 tiles, the last 64 channels, 32 per group
    # 65..128 channels on rows of 130..256 columns: a unit of one row, a quarter band
    "c5_co128_w200": W["c5_gn_pool_clamp"].resized(N=1, H=13, W=200, Cout=128, groups=16),  # stats-only rows
    "c5_co96_w256": W["c5_gn_pool_clamp"].resized(N=2, H=9, W=256, Cout=96, groups=12),     # 32 zero filters, 63 windows
    # rows wider than 256 fused (Cout <= 64): column tiles of 252 outputs
    "c5_w300": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=300),                   # last tile 46 columns: both passes masked
    "c5_w510": W["c5_gn_pool_clamp"].resized(N=1, H=9, W=510, Cout=32, groups=8),  # 3 tiles, the last one window, a stats-only row
    # more than 128 channels fused: channel tiles of 128, each unit one tile's half band
    "c5_co256_w128": W["c5_gn_pool_clamp"].resized(N=2, H=13, W=128, Cout=256, groups=32),  # 2 tiles, a stats-only row
    "c5_co200_w100": W["c5_gn_pool_clamp"].resized(N=1, H=14, W=100, Cout=200, groups=25),  # last tile 72 channels
    "c5_co384_w80": W["c5_gn_pool_clamp"].resized(N=1, H=10, W=80, Cout=384, groups=6),     # 3 tiles, 64 per group, P 80
}
FP32_ONLY = {"c2wide": W["c2_min_tanh2"].resized(N=1, H=6, W=300)}       # row wider than one tile
# shapes the tf32 kernel refuses: the call must say so, not fall back
TF32_REFUSED = set()


def modes():
    import x3_conv2d_epilogue_gb300 as ce
    return {"fp32": ce.MODE_FP32, "tf32": ce.MODE_TF32}


@pytest.mark.parametrize("mode", ["fp32", "tf32"])
@pytest.mark.parametrize("case", sorted(SMALL))
def test_small_parity(case, mode):
    wl = SMALL[case]
    t = synth.make_inputs(wl, seed=0)
    m = modes()[mode]
    if mode == "tf32" and case in TF32_REFUSED:
        import x3_conv2d_epilogue_gb300 as ce
        with pytest.raises(ce.ConvEpiError) as info:
            gpu_run(wl, t, m)
        assert ce.STATUS[info.value.status] == "UNSUPPORTED"
        return
    got, idx = gpu_run(wl, t, m, want_index=(mode == "fp32" and fp32_indices(wl)))
    ref, ref_idx = oracle_run(wl, t)
    if mode == "fp32":
        check_fp32(got, ref, case)
    else:
        check_tf32(got, ref, case)
    if idx is not None:
        y = oracle.conv3x3(t.x, t.w, t.b)
        if wl.kind == synth.KIND_GN_SCALE_POOL_CLAMP:
            sign = np.sign(t.gamma.astype(np.float64) * t.scale)[None, :].repeat(wl.N, 0)
            gap = pool_index_gap(y, wl.pool_k, np.where(sign >= 0, 1.0, -1.0)) * np.abs(
                (t.gamma.astype(np.float64) * t.scale))[None, :, None, None]
        else:
            gap = min_index_gap(y, wl.scalar)
        check_index(idx, ref_idx, gap, case)


@pytest.mark.parametrize("case", sorted(FP32_ONLY))
def test_fp32_only_shapes(case):
    import x3_conv2d_epilogue_gb300 as ce
    wl = FP32_ONLY[case]
    t = synth.make_inputs(wl, seed=1)
    got, idx = gpu_run(wl, t, ce.MODE_FP32, want_index=True)
    ref, ref_idx = oracle_run(wl, t)
    check_fp32(got, ref, case)
    check_index(idx, ref_idx, min_index_gap(oracle.conv3x3(t.x, t.w, t.b), wl.scalar), case)


@pytest.mark.parametrize("mode", ["fp32", "tf32"])
@pytest.mark.parametrize("case", ["pr1", "c4s", "c2s"])
def test_integer_inputs_bit_exact(case, mode):
    """Integer x, w, b with |v| <= 8: every product and partial sum is an
    integer below 2^24 and every operand fits tf32, so the conv is exact in
    both modes and the min chain's value must match to the last bit."""
    wl = SMALL[case]
    t = synth.make_integer_inputs(wl, seed=3)
    got, _ = gpu_run(wl, t, modes()[mode])
    y = oracle.conv3x3(t.x, t.w, t.b)
    ref, _ = oracle.chain_min(y, wl.scalar, wl.kind == synth.KIND_MIN_TANH2)
    if wl.kind == synth.KIND_SCALE_MIN:
        np.testing.assert_array_equal(got.astype(np.float64), ref)
    else:
        # tanh(tanh(integer)): the fp32 tanhf of an exact argument
        np.testing.assert_allclose(got, ref, rtol=0, atol=2e-7)


@pytest.mark.parametrize("mode", ["fp32", "tf32"])
def test_delta_kernel_reproduces_input(mode):
    """Centre-tap identity filter + per-channel chain with multiplier 1 and
    slope 1: out = GELU(x cropped), to within the mode's tolerance."""
    wl = W["c3_mul_lrelu_gelu"].resized(N=1, H=9, lrelu_slope=1.0)
    t = synth.make_inputs(wl, seed=5)
    t.w[:] = 0
    for co in range(wl.Cout):
        t.w[co, co % wl.Cin, 1, 1] = 1.0
    t.b[:] = 0
    t.mult[:] = 1.0
    got, _ = gpu_run(wl, t, modes()[mode])
    ref, _ = oracle_run(wl, t)
    xc = t.x[:, np.arange(wl.Cout) % wl.Cin, 1:-1, 1:-1].astype(np.float64)
    gelu = 0.5 * xc * (1 + np.vectorize(__import__("math").erf)(xc / np.sqrt(2)))
    np.testing.assert_allclose(ref, gelu, rtol=1e-12, atol=1e-12)
    (check_fp32 if mode == "fp32" else check_tf32)(got, ref, "delta")


def test_repeated_forward_is_deterministic():
    import x3_conv2d_epilogue_gb300 as ce
    wl = SMALL["c5t"]
    t = synth.make_inputs(wl, seed=9)
    a, _ = gpu_run(wl, t, ce.MODE_FP32, repeats=1)
    b, _ = gpu_run(wl, t, ce.MODE_FP32, repeats=3)
    np.testing.assert_array_equal(a, b)


def tf32_rna(x: np.ndarray) -> np.ndarray:
    """fp32 -> tf32 by the rounding rule of the tensor-core mode: keep 10
    mantissa bits, round to nearest with ties away from zero (finite values)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x1000) & 0xFFFFE000).astype(np.uint32)
    return r.view(np.float32)


def test_tf32_operand_rounding_is_exact():
    """tf32 mode with a centre-tap filter on one channel and every other
    channel biased far above it: the channel minimum is that channel's
    y = tf32(x) * 1, an exact product and a single-term sum, so the output must
    equal the rounded input bit for bit.  Inputs include exact ties (dropped
    bits 0x1000) of both signs, values one below and one above a tie, and
    values whose rounding carries into the exponent."""
    import x3_conv2d_epilogue_gb300 as ce
    wl = W["c4_scale_min"].resized(N=1, Cin=8, H=6, W=32, Cout=64, scalar=1.0)
    t = synth.make_inputs(wl, seed=11)
    rng = np.random.default_rng(3)
    bits = rng.normal(size=t.x.shape).astype(np.float32).view(np.uint32)
    flat = bits.reshape(-1)
    special = np.array([0x1000, 0x0FFF, 0x1001, 0x1FFF, 0x2000], dtype=np.uint32)
    flat[:] = (flat & 0xFFFFE000) | special[np.arange(flat.size) % special.size]
    flat[::7] |= 0x80000000                          # both signs on the tie patterns
    flat[5::11] = (flat[5::11] & 0x80000000) | 0x3F7FF000   # rounds up into the next binade
    t.x[:] = bits.view(np.float32)
    t.w[:] = 0
    t.w[0, 3, 1, 1] = 1.0
    t.b[:] = 1.0e6
    t.b[0] = 0.0
    got, _ = gpu_run(wl, t, ce.MODE_TF32)
    want = tf32_rna(t.x[:, 3:4, 1:-1, 1:-1])
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("case", sorted(SMALL))
def test_channels_last_parity(case):
    """The tf32 path with channels-last input: the same seeded values,
    transposed, against the same oracle and bound.  Shapes whose Cin is not a
    multiple of 4 are refused with UNSUPPORTED."""
    import x3_conv2d_epilogue_gb300 as ce
    wl = SMALL[case]
    t = synth.make_inputs(wl, seed=0)
    if wl.Cin % 4 != 0 or case in TF32_REFUSED:
        with pytest.raises(ce.ConvEpiError) as info:
            gpu_run(wl, t, ce.MODE_TF32, layout=ce.LAYOUT_NHWC)
        assert ce.STATUS[info.value.status] == "UNSUPPORTED"
        return
    got, _ = gpu_run(wl, t, ce.MODE_TF32, layout=ce.LAYOUT_NHWC)
    check_tf32(got, oracle_run(wl, t)[0], case + " nhwc")


def tf32_trunc(x: np.ndarray) -> np.ndarray:
    """fp32 -> the top 19 bits (sign, exponent, 10 mantissa bits): truncation
    toward zero of the low 13 mantissa bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (u & np.uint32(0xFFFFE000)).view(np.float32)


def test_channels_last_operands_are_truncated():
    """Channels-last input reaches the tensor core without a rounding pass:
    with a centre-tap filter on one channel and every other channel biased
    far above it, the channel minimum is that channel's y = x * 1 with x cut
    to its top 19 bits, bit for bit (the same inputs as the rounding test,
    whose tie patterns tell truncation from rounding)."""
    import x3_conv2d_epilogue_gb300 as ce
    wl = W["c4_scale_min"].resized(N=1, Cin=8, H=6, W=32, Cout=64, scalar=1.0)
    t = synth.make_inputs(wl, seed=11)
    rng = np.random.default_rng(3)
    bits = rng.normal(size=t.x.shape).astype(np.float32).view(np.uint32)
    flat = bits.reshape(-1)
    special = np.array([0x1000, 0x0FFF, 0x1001, 0x1FFF, 0x2000], dtype=np.uint32)
    flat[:] = (flat & 0xFFFFE000) | special[np.arange(flat.size) % special.size]
    flat[::7] |= 0x80000000
    t.x[:] = bits.view(np.float32)
    t.w[:] = 0
    t.w[0, 3, 1, 1] = 1.0
    t.b[:] = 1.0e6
    t.b[0] = 0.0
    got, _ = gpu_run(wl, t, ce.MODE_TF32, layout=ce.LAYOUT_NHWC)
    want = tf32_trunc(t.x[:, 3:4, 1:-1, 1:-1])
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))


def test_fp32_two_pass_groupnorm_refuses_indices():
    """The fp32 mode runs GroupNorm shapes its kernel does not take (here
    3 x 3 windows, and 128 groups) as the conv then the chain's post-pass,
    which computes no window indices: asking for them is UNSUPPORTED, while
    the same shapes without indices match the oracle (test_small_parity)."""
    import x3_conv2d_epilogue_gb300 as ce
    for wl in (SMALL["c5_k3"], SMALL["c5_co128_g128"]):
        t = synth.make_inputs(wl, seed=0)
        with pytest.raises(ce.ConvEpiError) as info:
            gpu_run(wl, t, ce.MODE_FP32, want_index=True)
        assert ce.STATUS[info.value.status] == "UNSUPPORTED"


CL_EXTRA = {
    "c4_cin100": W["c4_scale_min"].resized(N=2, H=6, W=40, Cin=100),   # span transpose, 32 positions a block, ragged last
    "c3_cin129": W["c3_mul_lrelu_gelu"].resized(N=1, H=5, W=37, Cin=129),   # tiled transpose, ragged tiles
}


@pytest.mark.parametrize("case", ["c2_w255", "c3_w67", "c5_w37", "c5_k3", "min_w3", "c4_w262", "c3cin3", "c4cin20",
                                  "c2cin12", "c2_cin256", "c4_cin100", "c3_cin129"])
def test_channels_last_fp32_matches_nchw(case):
    """The fp32 mode with channels-last input: an on-device transpose to
    NCHW, then the same kernel, so values and indices equal the NCHW run's
    bit for bit (any Cin; the tensor-core path needs Cin a multiple of 4).
    At most 128 channels go through the span transpose, more through 32 x 32
    tiles."""
    import x3_conv2d_epilogue_gb300 as ce
    wl = SMALL.get(case) or CL_EXTRA[case]
    t = synth.make_inputs(wl, seed=3)
    want_index = fp32_indices(wl)
    ref, ref_idx = gpu_run(wl, t, ce.MODE_FP32, want_index=want_index)
    got, idx = gpu_run(wl, t, ce.MODE_FP32, want_index=want_index, layout=ce.LAYOUT_NHWC)
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))
    check_fp32(got, oracle_run(wl, t)[0], case)
    if want_index:
        np.testing.assert_array_equal(idx, ref_idx)


@pytest.mark.parametrize("case", ["c5s", "c5t", "c5_w37", "c5_k2", "c5_k1", "c5g1", "c5_cin20"])
def test_fp32_groupnorm_values_do_not_depend_on_indices(case):
    """The fp32 GroupNorm kernel tracks window indices only when index_out is
    given; without it it keeps the extremes as values alone.  Both give the
    same outputs bit for bit."""
    import x3_conv2d_epilogue_gb300 as ce
    wl = SMALL[case]
    t = synth.make_inputs(wl, seed=5)
    with_idx, _ = gpu_run(wl, t, ce.MODE_FP32, want_index=True)
    without, _ = gpu_run(wl, t, ce.MODE_FP32, want_index=False)
    np.testing.assert_array_equal(without.view(np.uint32), with_idx.view(np.uint32))
    check_fp32(without, oracle_run(wl, t)[0], case)
