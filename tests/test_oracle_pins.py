"""Pins of the fp64 oracle against things other than itself.

Each test ties one oracle function to a library routine (torch CPU fp64
conv2d / group_norm / max_pool2d / gelu / leaky_relu, numpy argmin), to brute
force on tiny tensors, to a closed form or to an invariant, so that a dropped
term, a wrong sign or index, or a transposed operand fails at least one of
them.  CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed):
    return np.random.default_rng(seed)


def rand(shape, seed, lo=-1.0, hi=1.0):
    return rng(seed).uniform(lo, hi, size=shape).astype(np.float32)


def torch_conv(x, w, b):
    return F.conv2d(torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                    torch.from_numpy(b).double()).numpy()


# --------------------------------------------------------------------------
# shapes (values the pages state)
# --------------------------------------------------------------------------
def read_golden_shapes():
    rows = []
    with open(os.path.join(GOLDEN, "shapes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                what, a, b = line.split()
                rows.append((what, int(a), int(b)))
    return rows


def test_golden_shapes():
    rows = read_golden_shapes()
    assert len(rows) == 4
    for what, a, b in rows:
        if what == "conv":
            assert oracle.conv_out(a, a) == (b, b)
        elif what == "pool4":
            assert oracle.pool_out(a, 4) == b
        else:
            raise AssertionError(what)


def read_golden_gn_counts():
    rows = []
    with open(os.path.join(GOLDEN, "gn_counts.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(tuple(int(v) for v in line.split()))
    return rows


def test_golden_gn_counts():
    """The oracle's GroupNorm statistics run over the element count the pages
    state.  One conv output of the group holds the count itself and every
    other one is zero (a centre-tap filter on one channel copies a single
    non-zero input), so the mean is exactly 1 only if the oracle divides by
    that count, and the biased variance is exactly count - 1."""
    rows = read_golden_gn_counts()
    assert len(rows) == 1
    for N, Cin, H, W, Cout, G, count, pairs in rows:
        assert N * G == pairs
        x = np.zeros((1, Cin, H, W), np.float32)
        x[0, 0, 1 + 37, 1 + 101] = count
        w = np.zeros((Cout, Cin, 3, 3), np.float32)
        w[0, 0, 1, 1] = 1.0
        b = np.zeros(Cout, np.float32)
        one = np.ones(Cout, np.float32)
        ch = oracle.chain(oracle.GN_SCALE_POOL_CLAMP, groups=G, eps=0.0, gamma=one, beta=b, scale=one, pool_k=4)
        _, _, mean, rstd = oracle.gn_group(x, w, b, ch, 0, 0, nthreads=4)
        assert mean == 1.0
        assert abs(rstd * np.sqrt(count - 1.0) - 1.0) < 1e-12


def test_golden_output_counts():
    """Element counts of the full-size outputs: the product of the oracle's
    output shape (the pages' printed figures disagree with one another and
    with their own shapes; the fixture cites them)."""
    rows = []
    with open(os.path.join(GOLDEN, "output_counts.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(line.split())
    assert len(rows) == 2
    for N, Cin, H, W, Cout, chain, count in rows:
        kind = {"min": oracle.MIN_TANH2, "gn_pool4": oracle.GN_SCALE_POOL_CLAMP}[chain]
        ch = oracle.chain(kind, groups=16, pool_k=4)
        shape = oracle.output_shape(int(N), int(Cin), int(H), int(W), int(Cout), ch)
        assert int(np.prod(shape)) == int(count)


def test_pool_out_matches_torch_floor_mode():
    for ho in range(4, 40):
        for k in (2, 3, 4, 5):
            if ho < k:
                continue
            t = F.max_pool2d(torch.zeros(1, 1, ho, ho), k)
            assert oracle.pool_out(ho, k) == t.shape[-1]


def test_output_shapes_per_chain():
    for wl in synth.WORKLOADS.values():
        t = synth.Tensors(None, None, None, np.ones(wl.Cout), np.ones(wl.Cout), np.zeros(wl.Cout), np.ones(wl.Cout))
        ch = oracle.chain_for(wl, t)
        shp = oracle.output_shape(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, ch)
        if wl.kind in (synth.KIND_MIN_TANH2, synth.KIND_SCALE_MIN):
            assert shp == (wl.N, 1, wl.H - 2, wl.W - 2)
        elif wl.kind == synth.KIND_MUL_LRELU_GELU:
            assert shp == (wl.N, wl.Cout, wl.H - 2, wl.W - 2)
        else:
            assert shp == (wl.N, wl.Cout, 31, 31)
    assert oracle.output_shape(2, 16, 32, 32, 64, oracle.chain(1)) == (2, 1, 30, 30)


# --------------------------------------------------------------------------
# conv core
# --------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(1, 1, 3, 3, 1), (2, 3, 7, 9, 5), (1, 8, 12, 10, 4), (3, 2, 5, 17, 3)])
def test_conv_matches_torch_fp64(shape):
    N, Cin, H, W, Cout = shape
    x = rand((N, Cin, H, W), 1)
    w = rand((Cout, Cin, 3, 3), 2)
    b = rand((Cout,), 3)
    y = oracle.conv3x3(x, w, b, nthreads=3)
    ref = torch_conv(x, w, b)
    assert y.shape == ref.shape
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)


def test_conv_integer_brute_force_exact():
    # pure-Python integer arithmetic on a tiny problem: exact equality
    N, Cin, H, W, Cout = 2, 2, 5, 6, 3
    g = rng(7)
    x = g.integers(-8, 9, size=(N, Cin, H, W)).astype(np.float32)
    w = g.integers(-8, 9, size=(Cout, Cin, 3, 3)).astype(np.float32)
    b = g.integers(-8, 9, size=(Cout,)).astype(np.float32)
    y = oracle.conv3x3(x, w, b)
    for n in range(N):
        for co in range(Cout):
            for i in range(H - 2):
                for j in range(W - 2):
                    s = int(b[co])
                    for ci in range(Cin):
                        for kh in range(3):
                            for kw in range(3):
                                s += int(w[co, ci, kh, kw]) * int(x[n, ci, i + kh, j + kw])
                    assert y[n, co, i, j] == s


def test_conv_delta_kernel_reproduces_cropped_input():
    N, Cin, H, W, Cout = 2, 3, 9, 11, 7
    x = rand((N, Cin, H, W), 11)
    w = np.zeros((Cout, Cin, 3, 3), np.float32)
    for co in range(Cout):
        w[co, co % Cin, 1, 1] = 1.0
    b = np.zeros(Cout, np.float32)
    y = oracle.conv3x3(x, w, b)
    for co in range(Cout):
        np.testing.assert_array_equal(y[:, co], x[:, co % Cin, 1:H - 1, 1:W - 1].astype(np.float64))


def test_conv_off_centre_delta_picks_the_right_tap():
    # a single 1 at (kh, kw) shifts the window by (kh, kw): catches swapped kh/kw
    N, Cin, H, W = 1, 1, 6, 8
    x = rand((N, Cin, H, W), 12)
    for kh in range(3):
        for kw in range(3):
            w = np.zeros((1, 1, 3, 3), np.float32)
            w[0, 0, kh, kw] = 1.0
            y = oracle.conv3x3(x, w, np.zeros(1, np.float32))
            np.testing.assert_array_equal(y[0, 0], x[0, 0, kh:kh + H - 2, kw:kw + W - 2])


def test_conv_constant_input_closed_form():
    N, Cin, H, W, Cout = 1, 4, 6, 5, 6
    c = 0.75
    x = np.full((N, Cin, H, W), c, np.float32)
    w = rand((Cout, Cin, 3, 3), 13)
    b = rand((Cout,), 14)
    y = oracle.conv3x3(x, w, b)
    expect = c * w.astype(np.float64).reshape(Cout, -1).sum(1) + b
    for co in range(Cout):
        np.testing.assert_allclose(y[0, co], expect[co], rtol=0, atol=1e-14)


def test_conv_channel_mixing_is_not_transposed():
    # w[co, ci] = 0 except one (co, ci) pair: only that output channel sees
    # only that input channel
    N, Cin, H, W, Cout = 1, 3, 5, 5, 4
    x = rand((N, Cin, H, W), 15)
    w = np.zeros((Cout, Cin, 3, 3), np.float32)
    w[3, 1] = rand((3, 3), 16)
    b = np.zeros(Cout, np.float32)
    y = oracle.conv3x3(x, w, b)
    assert np.all(y[0, :3] == 0)
    ref = torch_conv(x[:, 1:2], w[3:4, 1:2], np.zeros(1, np.float32))
    np.testing.assert_allclose(y[0, 3], ref[0, 0], rtol=1e-14, atol=1e-14)


# --------------------------------------------------------------------------
# min chains
# --------------------------------------------------------------------------
@pytest.mark.parametrize("scalar,tanh2", [(1.0, True), (2.0, False), (-1.5, False), (0.5, True)])
def test_min_chain_matches_torch(scalar, tanh2):
    y = rng(21).normal(size=(2, 9, 4, 5))
    out, arg = oracle.chain_min(y, scalar=scalar, tanh2=tanh2)
    t = torch.from_numpy(y) * scalar
    ref = torch.min(t, dim=1, keepdim=True)[0]
    if tanh2:
        ref = torch.tanh(torch.tanh(ref))
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-15, atol=1e-15)
    np.testing.assert_array_equal(arg[:, 0], np.argmin(scalar * y, axis=1))


def test_min_chain_ties_keep_first_channel():
    y = np.zeros((1, 5, 1, 3))
    y[0, :, 0, 0] = [3, 1, 2, 1, 1]
    y[0, :, 0, 1] = [-4, -4, 0, 0, -4]
    y[0, :, 0, 2] = [2, 2, 2, 2, 2]
    _, arg = oracle.chain_min(y, 1.0, False)
    assert arg[0, 0, 0].tolist() == [1, 0, 0]


def test_tanh2_bounds_and_oddness():
    y = rng(22).normal(scale=5, size=(1, 4, 8, 8))
    out, _ = oracle.chain_min(y, 1.0, True)
    assert np.all(np.abs(out) < math.tanh(1.0))
    out_neg, _ = oracle.chain_min(-y, -1.0, True)   # min(-1 * -y) = min(y)
    np.testing.assert_array_equal(out_neg, out)
    # odd function: tanh(tanh(-m)) = -tanh(tanh(m)) where m = min(y) = -max(-y)
    out_flip, _ = oracle.chain_min(-y, 1.0, True)   # tanh2(min(-y)) = tanh2(-max(y))
    ref = -np.tanh(np.tanh(y.max(axis=1, keepdims=True)))
    np.testing.assert_allclose(out_flip, ref, rtol=1e-15, atol=1e-15)


# --------------------------------------------------------------------------
# per-channel chain: x mult -> LeakyReLU -> erf GELU
# --------------------------------------------------------------------------
def test_mul_lrelu_gelu_matches_torch():
    y = rng(31).normal(scale=3, size=(2, 6, 5, 4))
    mult = rand((6,), 32, -2, 2)
    out = oracle.chain_mul_lrelu_gelu(y, mult, 0.01)
    t = torch.from_numpy(y) * torch.from_numpy(mult.astype(np.float64)).view(1, -1, 1, 1)
    ref = F.gelu(F.leaky_relu(t, 0.01), approximate="none")
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-14, atol=1e-15)


def test_gelu_identities():
    # slope 1 makes LeakyReLU the identity and mult 1 leaves y: out = GELU(y)
    v = np.linspace(-8, 8, 161).reshape(1, 1, 1, -1)
    ones = np.ones(1, np.float32)
    g = oracle.chain_mul_lrelu_gelu(v, ones, 1.0)
    gneg = oracle.chain_mul_lrelu_gelu(-v, ones, 1.0)
    np.testing.assert_allclose(gneg, g - v, rtol=0, atol=1e-14)        # GELU(-x) = GELU(x) - x
    assert oracle.chain_mul_lrelu_gelu(np.zeros((1, 1, 1, 1)), ones, 1.0)[0, 0, 0, 0] == 0.0
    big = v[v > 6.0]
    gb = oracle.chain_mul_lrelu_gelu(big.reshape(1, 1, 1, -1), ones, 1.0).ravel()
    assert np.all(np.abs(gb - big) < 1e-8 * big)                       # GELU(x) ~ x for x > 6
    # x * Phi(x) with Phi from the closed form of the normal CDF via erfc
    phi = 0.5 * np.array([math.erfc(-t / math.sqrt(2)) for t in v.ravel()])
    np.testing.assert_allclose(g.ravel(), v.ravel() * phi, rtol=1e-13, atol=1e-15)


def test_leaky_relu_slope_applies_to_negatives_only():
    v = np.array([-2.0, -0.5, 0.0, 0.5, 2.0]).reshape(1, 1, 1, -1)
    ones = np.ones(1, np.float32)
    out = oracle.chain_mul_lrelu_gelu(v, ones, 0.01)
    lr = np.where(v > 0, v, 0.01 * v)
    ref = 0.5 * lr * (1 + np.vectorize(math.erf)(lr / math.sqrt(2)))
    np.testing.assert_allclose(out, ref, rtol=1e-15, atol=1e-18)


# --------------------------------------------------------------------------
# GroupNorm -> scale -> max-pool -> clamp
# --------------------------------------------------------------------------
def gn_ref_torch(y, groups, gamma, beta, scale, k, lo, hi, eps=1e-5):
    t = torch.from_numpy(y)
    g = F.group_norm(t, groups, torch.from_numpy(gamma.astype(np.float64)),
                     torch.from_numpy(beta.astype(np.float64)), eps)
    g = g * torch.from_numpy(scale.astype(np.float64)).view(1, -1, 1, 1)
    return F.max_pool2d(g, k).clamp(lo, hi).numpy(), g.numpy()


@pytest.mark.parametrize("Ho,k", [(14, 4), (13, 3), (9, 2)])
def test_gn_pool_matches_torch(Ho, k):
    N, C, G = 2, 8, 4
    y = rng(41).normal(loc=0.3, scale=2.0, size=(N, C, Ho, Ho + 1))
    gamma = rand((C,), 42, 0.5, 1.5)
    beta = rand((C,), 43, -0.3, 0.3)
    scale = rand((C,), 44, -1.0, 2.0)          # some negative channels
    ch = oracle.chain(oracle.GN_SCALE_POOL_CLAMP, groups=G, eps=1e-5, gamma=gamma, beta=beta, scale=scale,
                      pool_k=k, clamp_lo=0.0, clamp_hi=1.0)
    out, arg, mean, rstd = oracle.chain_gn_pool(y, ch)
    ref, normed = gn_ref_torch(y, G, gamma, beta, scale, k, 0.0, 1.0)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    # statistics: biased variance over (C/G, H, W) of each (n, g)
    yg = y.reshape(N, G, -1)
    np.testing.assert_allclose(mean, yg.mean(-1), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(rstd, 1 / np.sqrt(yg.var(-1) + 1e-5), rtol=1e-12)
    # index = first row-major position of the window maximum of the normalised value
    Hp = out.shape[2]
    Wp = out.shape[3]
    for n in range(N):
        for c in range(C):
            for ph in range(Hp):
                for pw in range(Wp):
                    win = normed[n, c, ph * k:ph * k + k, pw * k:pw * k + k].ravel()
                    assert arg[n, c, ph, pw] == int(np.argmax(win))


def test_gn_pre_affine_mean_zero_var_one():
    # gamma 1, beta 0, scale 1, pool 1, no clamp: out is the normalised tensor
    N, C, G, Ho = 2, 8, 2, 10
    y = rng(45).normal(loc=-0.7, scale=3.0, size=(N, C, Ho, Ho))
    one = np.ones(C, np.float32)
    ch = oracle.chain(oracle.GN_SCALE_POOL_CLAMP, groups=G, eps=1e-5, gamma=one, beta=np.zeros(C, np.float32),
                      scale=one, pool_k=1, clamp_lo=-1e300, clamp_hi=1e300)
    out, _, _, _ = oracle.chain_gn_pool(y, ch)
    z = out.reshape(N, G, -1)
    v = y.reshape(N, G, -1).var(-1)
    np.testing.assert_allclose(z.mean(-1), 0.0, atol=1e-12)
    np.testing.assert_allclose(z.var(-1), v / (v + 1e-5), rtol=1e-12)


def test_gn_stats_include_rows_the_pool_drops():
    # rows/cols 12..13 of a 14-wide map are outside every 4x4 window but must
    # still move the statistics
    N, C, G, Ho = 1, 4, 1, 14
    y = rng(46).normal(size=(N, C, Ho, Ho))
    y2 = y.copy()
    y2[:, :, 12:, :] += 5.0
    one = np.ones(C, np.float32)
    mk = lambda: oracle.chain(oracle.GN_SCALE_POOL_CLAMP, groups=G, gamma=one, beta=np.zeros(C, np.float32),
                              scale=one, pool_k=4, clamp_lo=-1e9, clamp_hi=1e9)
    o1, _, m1, _ = oracle.chain_gn_pool(y, mk())
    o2, _, m2, _ = oracle.chain_gn_pool(y2, mk())
    assert m2[0, 0] > m1[0, 0]
    assert not np.allclose(o1, o2)


def test_gn_negative_scale_turns_max_into_min():
    N, C, G, Ho, k = 1, 4, 2, 8, 4
    y = rng(47).normal(size=(N, C, Ho, Ho))
    one = np.ones(C, np.float32)
    zero = np.zeros(C, np.float32)
    mk = lambda s: oracle.chain(oracle.GN_SCALE_POOL_CLAMP, groups=G, gamma=one, beta=zero, scale=s, pool_k=k,
                                clamp_lo=-1e9, clamp_hi=1e9)
    pos, _, _, _ = oracle.chain_gn_pool(y, mk(one))
    neg, _, _, _ = oracle.chain_gn_pool(y, mk(-one))
    # with scale -1 the pooled value is -(window minimum of the normalised map)
    _, normed = gn_ref_torch(y, G, one, zero, one, 1, -1e9, 1e9)
    mins = -torch.from_numpy(-normed).unfold(2, k, k).unfold(3, k, k).amax((-1, -2)).numpy()
    np.testing.assert_allclose(neg, -mins, rtol=1e-13, atol=1e-13)
    assert not np.allclose(pos, neg)


def test_clamp_bounds():
    N, C, G, Ho = 1, 8, 4, 12
    y = rng(48).normal(scale=4, size=(N, C, Ho, Ho))
    beta = np.array([-6, -6, 0, 0, 0.5, 0.5, 6, 6], np.float32)   # some channels pinned at 0, some at 1
    gamma, scale = rand((C,), 1, 0.5, 2), rand((C,), 3, 0.5, 2)
    ch = oracle.chain(oracle.GN_SCALE_POOL_CLAMP, groups=G, gamma=gamma, beta=beta, scale=scale, pool_k=4,
                      clamp_lo=0.0, clamp_hi=1.0)
    out, _, _, _ = oracle.chain_gn_pool(y, ch)
    assert out.min() >= 0.0 and out.max() <= 1.0
    assert (out == 0.0).any() and (out == 1.0).any() and ((out > 0) & (out < 1)).any()
    ref, _ = gn_ref_torch(y, G, gamma, beta, scale, 4, 0.0, 1.0)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# whole forward and sampled evaluators agree with the composed pieces
# --------------------------------------------------------------------------
def small_workloads():
    return [
        synth.WORKLOADS["pr1_min_tanh2"],
        synth.WORKLOADS["c4_scale_min"].resized(N=2, Cin=8, H=9, W=12, Cout=16),
        synth.WORKLOADS["c3_mul_lrelu_gelu"].resized(N=2, Cin=8, H=10, W=9, Cout=8),
        synth.WORKLOADS["c5_gn_pool_clamp"].resized(N=2, Cin=8, H=18, W=14, Cout=16, groups=4),
    ]


@pytest.mark.parametrize("wl", small_workloads(), ids=lambda w: w.name)
def test_forward_equals_composition(wl):
    t = synth.make_inputs(wl, seed=0)
    ch = oracle.chain_for(wl, t)
    out, arg = oracle.forward(t.x, t.w, t.b, ch, nthreads=4)
    y = oracle.conv3x3(t.x, t.w, t.b)
    if wl.kind in (synth.KIND_MIN_TANH2, synth.KIND_SCALE_MIN):
        ref, rarg = oracle.chain_min(y, wl.scalar, wl.kind == synth.KIND_MIN_TANH2)
        np.testing.assert_array_equal(arg, rarg)
    elif wl.kind == synth.KIND_MUL_LRELU_GELU:
        ref = oracle.chain_mul_lrelu_gelu(y, t.mult, wl.lrelu_slope)
    else:
        ref, rarg, _, _ = oracle.chain_gn_pool(y, ch)
        np.testing.assert_array_equal(arg, rarg)
    np.testing.assert_array_equal(out, ref)


def test_sampled_evaluators_agree_with_forward():
    g = rng(51)
    wl = small_workloads()[1]
    t = synth.make_inputs(wl)
    out, arg = oracle.forward(t.x, t.w, t.b, oracle.chain_for(wl, t))
    n, i, j = (g.integers(0, s, 20) for s in (wl.N, wl.H - 2, wl.W - 2))
    o, a = oracle.min_at(t.x, t.w, t.b, n, i, j, scalar=wl.scalar, tanh2=False)
    np.testing.assert_array_equal(o, out[n, 0, i, j])
    np.testing.assert_array_equal(a, arg[n, 0, i, j])

    wl = small_workloads()[2]
    t = synth.make_inputs(wl)
    out, _ = oracle.forward(t.x, t.w, t.b, oracle.chain_for(wl, t))
    n, co, i, j = (g.integers(0, s, 20) for s in (wl.N, wl.Cout, wl.H - 2, wl.W - 2))
    o = oracle.mul_lrelu_gelu_at(t.x, t.w, t.b, t.mult, n, co, i, j)
    np.testing.assert_array_equal(o, out[n, co, i, j])

    wl = small_workloads()[3]
    t = synth.make_inputs(wl)
    ch = oracle.chain_for(wl, t)
    out, arg = oracle.forward(t.x, t.w, t.b, ch)
    cpg = wl.Cout // wl.groups
    for n in range(wl.N):
        for gi in range(wl.groups):
            o, a, _, _ = oracle.gn_group(t.x, t.w, t.b, ch, n, gi, nthreads=3)
            np.testing.assert_array_equal(o, out[n, gi * cpg:(gi + 1) * cpg])
            np.testing.assert_array_equal(a, arg[n, gi * cpg:(gi + 1) * cpg])


def test_conv_at_matches_torch_on_workload_shapes():
    wl = synth.WORKLOADS["c5_gn_pool_clamp"].resized(N=1)
    t = synth.make_inputs(wl)
    ref = torch_conv(t.x[:, :, :8, :8], t.w, t.b)
    for (co, i, j) in [(0, 0, 0), (63, 5, 5), (17, 2, 4)]:
        assert abs(oracle.conv_at(t.x, t.w, t.b, 0, co, i, j) - ref[0, co, i, j]) < 1e-13
