"""The tensor-core kernel's index ranges, checked on the CPU.

conv_epi_plan_query returns the plan a forward would launch (a pure host
call).  For every shape the GPU tests run, the full-size workloads and a
seeded sweep of random shapes, these tests check that every access the
kernel's roles make from that plan stays inside its buffer: the tensor-load
box and strides follow the 16-byte rules, column tiles start on 16-byte
boundaries, the shared-memory regions are disjoint and fit, the MMAs' filter
and input operand ranges stay inside their stages, the accumulators fit the
tensor memory, and the epilogue scratch holds what the chain stores there.
The access formulas below restate, from the kernel's roles, which rows and
bytes each MMA reads.
"""
import math
import random

import pytest

import synth
import x3_conv2d_epilogue_gb300 as ce

MIN_KINDS = (ce.MIN_TANH2, ce.SCALE_MIN)


def epi_for(kind, groups=16, pool_k=4):
    # the chain's parameter tensors are never read by a plan query: any
    # non-null value passes the argument checks
    return ce.epilogue(kind, chan_scale=16, gamma=16, beta=16, groups=groups, pool_k=pool_k)


def plan(N, Cin, H, W, Cout, kind, layout=ce.LAYOUT_NCHW, groups=16, pool_k=4):
    return ce.conv_epi_plan_query(N, Cin, H, W, Cout, epi_for(kind, groups, pool_k), layout)


def check_plan(q, N, Cin, H, W, Cout, kind, layout, pool_k=4):
    Ho, Wo = H - 2, W - 2
    nhwc = layout == ce.LAYOUT_NHWC
    S, P, U, RU, Rin, PL = q["S"], q["P"], q["U"], q["RU"], q["Rin"], q["PL"]
    # the GEMM: 64 or 128 output channels per tile, rows stacked into 128 lanes
    assert q["gemm_cout"] in (64, 128) and S * q["gemm_cout"] == 128
    assert q["gemm_cout"] == (64 if Cout <= 64 else 128)
    assert q["MT"] == (1 if Cout <= 128 else math.ceil(Cout / 128))
    assert q["chunks"] == math.ceil(Cin / 8)
    # MMA shape (kind::tf32, M = 128): N a multiple of 16 in 16 .. 256
    assert P % 16 == 0 and 16 <= P <= 256
    # rows of a unit; the tensor-load box height is at most 256
    assert RU == U * S and Rin == RU + 2 and Rin <= 256
    row_blocks = math.ceil(Ho / RU)
    assert q["units_per_image"] == row_blocks * q["CT"] * q["MT"]
    # tensor memory: U row sets of ucol >= P columns per buffer, two buffers
    assert q["ucol"] >= P and q["ucol"] % 32 == 0 and U * q["ucol"] <= q["acc_cols"]
    assert 2 * q["acc_cols"] <= q["tmem_cols"] <= 512
    # column tiles: every output column is covered once; tile starts are
    # 16-byte aligned (the tensor load's x coordinate) and a tile's inputs
    # (CW + 2 columns) fit the staged row
    CT, CW, BW = q["CT"], q["CW"], q["BW"]
    if CT == 1:
        assert CW == Wo and Wo <= P
        if not nhwc:
            assert BW >= W and BW % 4 == 0 and BW <= P
    else:
        assert BW == 256 and P == 256 and CW + 2 <= BW
        assert (CT - 1) * CW < Wo <= CT * CW
        for ct in range(CT):
            assert (ct * CW * 4) % 16 == 0
    # the tensor load: 16-byte inner box extent and strides, dims <= 256
    box = q["box"]
    assert all(1 <= v <= 256 for v in box)
    assert (box[0] * 4) % 16 == 0
    if nhwc:
        assert box == [4, P, Rin, 1] and (Cin * 4) % 16 == 0
        assert q["nr"] == 0 and q["raw_bytes"] == 0
        # two boxes of 4 channels x P positions x Rin rows land in one B plane
        assert Rin * P <= PL
    else:
        assert box == [BW, Rin, 8, 1]
        assert q["x_pitch"] >= W and (q["x_pitch"] * 4) % 16 == 0
        assert q["x_pitch"] == (W if W % 4 == 0 else W + (-W) % 4)
        assert q["raw_bytes"] >= 8 * Rin * BW * 4 and q["nr"] >= 2
        # converter: 2 * Rin * ceil(P / 32) items per chunk, within capacity;
        # it writes plane rows rr * P + w (rr < Rin, w < P) of each group
        assert 2 * Rin * math.ceil(P / 32) <= q["conv_items"]
        assert Rin * P <= PL
    # B operand: accumulator row set u, shift sk (0 .. S+1) and tap kw read P
    # rows starting at (u*S + sk)*P + kw of each 4-channel group
    top = max((u * S + sk) * P + kw + P for u in range(U) for sk in range(S + 2) for kw in range(3))
    assert top <= PL and q["b_bytes"] >= 2 * PL * 16
    # A operand: shift sk and tap kw start at plane S+1-sk, tap block kw, and
    # read 128 rows of 16 bytes from each of the two K groups (a_lbo apart)
    ap, lbo, kws = q["a_plane_bytes"], q["a_lbo"], q["a_kw_stride"]
    assert ap == q["gemm_cout"] * 16 and lbo == (2 * S + 1) * ap and kws == 2 * lbo
    for sk in range(S + 2):
        for kw in range(3):
            for g in range(2):
                start = (S + 1 - sk) * ap + kw * kws + g * lbo
                assert start >= 0 and start + 128 * 16 <= q["a_bytes"]
    assert q["a_bytes"] % 1024 == 0 and q["b_bytes"] % 1024 == 0 and q["raw_bytes"] % 1024 == 0
    # the packed filter: the pack kernel writes, and the producer copies,
    # chunk c of channel tile m at (m * chunks + c) * a_bytes
    assert q["wpack_bytes"] >= q["MT"] * q["chunks"] * q["a_bytes"]
    # the padded copy of x: rows of x_pitch floats, one per (image, channel, row)
    if not nhwc and W % 4:
        assert q["xpad_bytes"] == N * Cin * H * q["x_pitch"] * 4
    else:
        assert q["xpad_bytes"] == 0
    # shared memory: filter (resident: every chunk), B planes, staged tiles,
    # scratch, barriers (last: the GroupNorm finalize reuses what lies below
    # them), in order and disjoint, within the CTA limit
    filt = (q["chunks"] * q["MT"] if q["resident"] else q["na"]) * q["a_bytes"]
    if q["resident"]:
        assert q["MT"] == 1 and q["na"] == 1
    else:
        assert 2 <= q["na"] <= 4
    assert 2 <= q["nb"] <= 4 and q["nr"] <= 4
    assert q["a_off"] == 0 and q["b_off"] >= filt
    assert q["raw_off"] >= q["b_off"] + q["nb"] * q["b_bytes"]
    assert q["scratch_off"] >= q["raw_off"] + q["nr"] * q["raw_bytes"]
    assert q["bar_off"] >= q["scratch_off"] + q["scratch_bytes"]
    assert q["smem"] >= q["bar_off"] + q["bar_bytes"] + 8
    assert q["smem"] <= q["smem_limit"] <= 232448
    assert q["b_off"] % 1024 == 0 and q["raw_off"] % 1024 == 0 and q["bar_off"] % 8 == 0
    assert q["scratch_off"] % 16 == 0
    # epilogue scratch: the min chains' per-(u, quadrant) partial rows, the
    # per-channel transpose tiles, the GroupNorm pooled tiles of each band
    if kind in MIN_KINDS:
        assert q["scratch_bytes"] >= U * 4 * P * 4
    elif kind in (ce.MUL_LRELU_GELU, ce.NONE):
        # a 32 x 16 staging tile per epilogue warp, read and written at
        # r * 16 + 4 * ((c / 4) ^ ((r / 2) & 3)) + c % 4 (r < 32, c < 16)
        top = max(r * 16 + 4 * ((c // 4) ^ ((r // 2) & 3)) + c % 4 for r in range(32) for c in range(16))
        assert top == 32 * 16 - 1 and q["scratch_bytes"] >= 8 * 32 * 16 * 4
    else:
        bands = U // 2
        assert (S == 2 and U in (2, 4) and P <= 128 and (P == 64 or W - 2 >= 64)) or \
            (S == 1 and U == 2 and 64 < P <= 128 and W - 2 >= 64) or (S == 1 and U == 4 and P == 64) or \
            (S == 2 and U == 1 and 128 < P <= 256 and W - 2 >= 127) or \
            (S == 1 and U == 1 and 128 < P <= 256 and W - 2 >= 128)  # (127: one column tile, both passes masked)
        if pool_k == 2:
            # 2 x 2 windows: two band regions of pitch 65 (up to 63 windows),
            # the statistics, 128-channel tables; the tile writes reach
            # (band * 2 + slot) * 64 * 65 + channel * 65 + window (window < 64)
            # (no stacking: one band, channel rows 0..127 of pitch 65; rows of
            # up to 64 columns: four bands of pitch 33, windows < 32)
            assert U in (1, 2, 4)
            if U == 1:
                # rows of 130..240 columns: one row pair, two slots of pitch 129 (windows < 128)
                top = max(sl * 64 * 129 + ch * 129 + w for sl in (0, 1) for ch in range(64) for w in range(128))
                assert top < 2 * 64 * 129 and q["scratch_bytes"] >= (2 * 64 * 129 + 2 * 256 + 2 * 128) * 4
            elif U == 4:
                top = max((b * 2 + sl) * 64 * 33 + ch * 33 + w for b in range(4) for sl in (0, 1) for ch in range(64)
                          for w in range(32))
                assert top < 4 * 2 * 64 * 33 and q["scratch_bytes"] >= (4 * 2 * 64 * 33 + 2 * 256 + 2 * 128) * 4
            else:
                top = max((b * 2 + sl) * 64 * 65 + ch * 65 + w for b in (0, 1) for sl in (0, 1) for ch in range(64)
                          for w in range(64))
                assert max(ch * 65 + w for ch in range(128) for w in range(64)) < top
                assert top < 2 * 2 * 64 * 65 and q["scratch_bytes"] >= (2 * 2 * 64 * 65 + 2 * 256 + 2 * 128) * 4
        elif U == 1:
            # wide rows: one band region of pitch 65 (up to 63 windows), the
            # statistics, 128-channel tables; the tile writes reach
            # slot * 64 * 65 + channel * 65 + window (window < 64)
            top = max(sl * 64 * 65 + ch * 65 + w for sl in (0, 1) for ch in range(64) for w in range(64))
            assert top < 2 * 64 * 65 and q["scratch_bytes"] >= (2 * 64 * 65 + 2 * 256 + 2 * 128) * 4
        else:
            # sign and bias tables: 64 channels (the page-shape kernel), else 128
            tables = 64 if Cout == 64 and (W <= 64 or W - 2 >= 96) else 128
            assert q["scratch_bytes"] >= (bands * 2 * 64 * 33 + 2 * 256 + 2 * tables) * 4


def parity_shapes():
    import test_conv_only_gpu as tn
    import test_parity_gpu as tp
    import test_zz_guard_gpu as tg
    shapes = dict(tp.SMALL)
    shapes.update(tp.FP32_ONLY)
    shapes.update({"none_" + k: v for k, v in tn.CASES.items()})
    shapes.update({"guard_" + k: v for k, v in tg.CASES.items()})
    for name, wl in synth.WORKLOADS.items():
        shapes["full_" + name] = wl
    return shapes


SHAPES = parity_shapes()


@pytest.mark.parametrize("case", sorted(SHAPES))
@pytest.mark.parametrize("layout", [ce.LAYOUT_NCHW, ce.LAYOUT_NHWC])
def test_plans_of_tested_shapes(case, layout):
    wl = SHAPES[case]
    args = (wl.N, wl.Cin, wl.H, wl.W, wl.Cout, wl.kind, layout)
    if layout == ce.LAYOUT_NHWC and wl.Cin % 4:
        with pytest.raises(ce.ConvEpiError) as ei:
            plan(*args, groups=wl.groups, pool_k=wl.pool_k)
        assert ce.STATUS[ei.value.status] == "UNSUPPORTED"
        return
    check_gn_form(plan(*args, groups=wl.groups, pool_k=wl.pool_k), *args, pool_k=wl.pool_k, groups=wl.groups)


def wide_p2_fits(Cin, W, nhwc):
    """2 x 2 windows on rows of 130..256 columns: the smallest plan (the
    filter resident when it fits beside 2 B planes and 2 staged tiles, else
    2 filter stages) with its two-slot tile of pitch 129 within the CTA's
    shared memory -- the kernel's own rule restated."""
    up1k = lambda v: (v + 1023) // 1024 * 1024
    P = (W + 15) // 16 * 16
    a = up1k(3 * 2 * 5 * 64 * 16)
    pl_ = (4 * P + 4 + 7) // 8 * 8
    b = up1k(2 * pl_ * 16)
    raw = 0 if nhwc else up1k(8 * 4 * ((W + 3) // 4 * 4) * 4)
    nr0 = 0 if nhwc else 2
    tail = 8 * 30 + 32 + (2 * 64 * 129 + 2 * 256 + 2 * 128) * 4
    chunks = (Cin + 7) // 8
    resident = chunks * a + 2 * b + nr0 * raw + tail <= 232448
    return (chunks * a if resident else 2 * a) + 2 * b + nr0 * raw + tail <= 232448


def gn_fused(kind, Cout, W, pool_k, groups, nhwc=False, Cin=8):
    # rows of up to 64 columns run as two pooling bands per unit; wider rows as
    # one band, fused when the first 96 output columns are whole (Wo >= 96);
    # up to 64 channels (a 64-channel GEMM), a group's channels a power of two
    # 65..128 channels (no row stacking) fuse with one-band rows, each unit
    # pooling half a band; one-band rows need Wo >= 64 (the generalised
    # kernel masks the chunks past column 64)
    cpg = Cout // groups
    if kind != ce.GN_SCALE_POOL_CLAMP or pool_k not in (2, 4) or cpg & (cpg - 1) or cpg > 64:
        return False
    if pool_k == 2:  # 2 x 2 windows: rows of up to 128 columns up to 128 channels, of 130..240 up to 64
        # (rows of 130..256: where the plan fits shared memory, e.g. W <= 240 for NCHW with Cin <= 8)
        return (Cout <= 128 and W <= 128 and W != 65) or (Cout <= 64 and 130 <= W <= 256 and wide_p2_fits(Cin, W, nhwc))
    # rows of 130..256 columns (Cout <= 64): one row pair per unit; wider
    # rows: the same per column tile of 252 outputs
    # more than 64 channels: no row stacking, half a band per unit (more than
    # 128: channel tiles of 128, a unit per tile)
    # (65..128 channels on rows of 130..256 columns: a quarter band per unit)
    return ((Cout <= 64 and (W <= 64 or W >= 66)) or (Cout > 64 and (W <= 64 or 66 <= W <= 128)) or
            (64 < Cout <= 128 and 130 <= W <= 256))


def check_gn_form(q, N, Cin, H, W, Cout, kind, layout, pool_k, groups):
    """A GroupNorm shape the fused epilogue does not take runs as two passes:
    its plan is the plain conv's, and the handle holds the conv output
    between them."""
    two_pass = kind == ce.GN_SCALE_POOL_CLAMP and not gn_fused(kind, Cout, W, pool_k, groups, layout == ce.LAYOUT_NHWC,
                                                               Cin)
    assert q["gn_two_pass"] == int(two_pass)
    # the conv output, then (256-byte aligned) the conv kernel's per-unit sums:
    # (image, unit, 2 column groups, 128 accumulator rows) float pairs
    if two_pass:
        ybytes = -(-(N * Cout * (H - 2) * (W - 2) * 4) // 256) * 256
        units = q["units_per_image"]
        assert q["ybuf_bytes"] == ybytes + N * units * 2 * 128 * 8
    else:
        assert q["ybuf_bytes"] == 0
    check_plan(q, N, Cin, H, W, Cout, ce.NONE if two_pass else kind, layout, pool_k)


def test_random_shapes_all_planned_and_in_range():
    """Every shape with H, W >= 3 has a plan (the tf32 mode takes any size),
    and every plan passes the range checks; GroupNorm shapes are fused
    exactly when groups have a power-of-two size up to 64 and either
    pool_k = 4 with Cout <= 64 and W != 65, or Cout > 64 with W <= 64 or
    66 <= W <= 128, or 64 < Cout <= 128 with 130 <= W <= 256, or pool_k = 2 with
    Cout <= 128 and W <= 128 (not 65) or Cout <= 64 and 130 <= W <= 256
    where the plan fits shared memory;
    otherwise they are planned as the plain
    conv of the two-pass form."""
    rng = random.Random(20261203)
    for _ in range(3000):
        kind = rng.choice([ce.MIN_TANH2, ce.SCALE_MIN, ce.MUL_LRELU_GELU, ce.GN_SCALE_POOL_CLAMP, ce.NONE])
        layout = rng.choice([ce.LAYOUT_NCHW, ce.LAYOUT_NHWC])
        N = rng.randint(1, 4)
        W = rng.choice([rng.randint(3, 40), rng.randint(41, 300), rng.randint(301, 1100)])
        H = rng.randint(3, 60)
        Cin = rng.choice([rng.randint(1, 24), rng.randint(25, 320)])
        Cout = rng.choice([rng.randint(1, 64), 64, rng.randint(65, 128), rng.randint(129, 400)])
        if layout == ce.LAYOUT_NHWC:
            Cin = max(4, Cin // 4 * 4)
        groups, pool_k = 1, 4
        if kind == ce.GN_SCALE_POOL_CLAMP:
            if rng.random() < 0.7:
                Cout, W = 64, rng.randint(6, 128)
            groups = rng.choice([g for g in (1, 2, 4, 8, 16, 32, 64) if Cout % g == 0] or [1])
            pool_k = rng.choice([4, 4, 4, 2])
            H = max(H, pool_k + 2)
            W = max(W, pool_k + 2)
        args = (N, Cin, H, W, Cout, kind, layout)
        check_gn_form(plan(*args, groups=groups, pool_k=pool_k), *args, pool_k=pool_k, groups=groups)


def test_plan_query_arguments():
    with pytest.raises(ce.ConvEpiError) as ei:          # fp32 mode has no tensor-core plan
        d = ce.Desc(1, 8, 8, 8, 64, ce.MODE_FP32, ce.LAYOUT_NCHW)
        q = ce.Plan()
        ce._check(ce._lib().conv_epi_plan_query(ce.C.byref(d), ce.C.byref(epi_for(ce.MIN_TANH2)),
                                                ce.C.byref(q)), "plan")
    assert ce.STATUS[ei.value.status] == "UNSUPPORTED"
    for bad_kind in (6, 7, 8, 9, 10, 11, 12, 13, 14, 15, -1):  # bad chain (the kernel's internal kinds included)
        with pytest.raises(ce.ConvEpiError) as ei:
            plan(1, 8, 8, 8, 64, bad_kind)
        assert ce.STATUS[ei.value.status] == "INVALID_ARG"
    with pytest.raises(ce.ConvEpiError) as ei:          # H < 3
        plan(1, 8, 2, 8, 64, ce.MIN_TANH2)
    assert ce.STATUS[ei.value.status] == "INVALID_ARG"
    assert ce._lib().conv_epi_plan_query(None, None, None) == 1
    q = plan(128, 16, 256, 256, 64, ce.MIN_TANH2)        # the C2 workload: one resident filter, one row tile
    assert q["struct_bytes"] == ce.C.sizeof(ce.Plan)
    assert (q["P"], q["U"], q["RU"], q["CT"], q["MT"], q["resident"]) == (256, 1, 2, 1, 1, 1)
