"""The seeded input generators that the oracle tests, the GPU parity tests and
the bench share: the generator matches its published definition, draws are
reproducible and addressable one element at a time (the sampled full-size
checks regenerate single elements), and the workload tensors have the stated
distributions.  CPU only."""
import math

import numpy as np

import synth


def test_splitmix64_reference_outputs():
    # the first outputs of SplitMix64 from state 1234567 in the generator's
    # reference C code (Vigna, splitmix64.c)
    got = synth.splitmix64(np.uint64(1234567), np.arange(5, dtype=np.uint64))
    assert [int(v) for v in got] == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                                     4593380528125082431, 16408922859458223821]


def test_draws_are_reproducible_and_seeded():
    wl = synth.WORKLOADS["c5_gn_pool_clamp"].resized(N=2, H=10, W=12)
    a, b, c = synth.make_inputs(wl, seed=0), synth.make_inputs(wl, seed=0), synth.make_inputs(wl, seed=1)
    for k in ("x", "w", "b", "gamma", "beta", "scale"):
        assert np.array_equal(getattr(a, k), getattr(b, k)), k
        assert not np.array_equal(getattr(a, k), getattr(c, k)), k
    # every tensor has its own stream: x and w of the same seed are unrelated
    assert not np.allclose(a.x.reshape(-1)[:16], a.w.reshape(-1)[:16])


def test_single_elements_regenerate():
    x = synth.normal((3, 5, 7), 0.0, 1.0, seed=4, stream=synth.STREAM_X)
    idx = np.array([0, 1, 17, 104], dtype=np.int64)
    np.testing.assert_array_equal(synth.normal_at(idx, 0.0, 1.0, seed=4, stream=synth.STREAM_X),
                                  x.reshape(-1)[idx].astype(np.float32))


def test_workload_distributions():
    wl = synth.WORKLOADS["c5_gn_pool_clamp"].resized(N=4, H=64, W=64)
    t = synth.make_inputs(wl, seed=0)
    for k in ("x", "w", "b", "gamma", "beta", "scale"):
        v = getattr(t, k)
        assert v.dtype == np.float32 and v.flags.c_contiguous, k
    assert abs(float(t.x.mean())) < 0.02 and abs(float(t.x.std()) - 1.0) < 0.02
    bound = 1.0 / math.sqrt(wl.Cin * 9)
    assert np.all(np.abs(t.w) <= bound) and np.all(np.abs(t.b) <= bound)
    assert abs(float(t.w.std()) - bound / math.sqrt(3.0)) < 0.1 * bound
    assert abs(float(t.gamma.mean()) - 1.0) < 0.05 and float(t.gamma.std()) < 0.2
    # scale ~ N(1, 0.5): some channels come out negative, which exercises the
    # pooled-minimum branch of the GroupNorm chain
    assert np.any(t.scale < 0) and abs(float(t.scale.mean()) - 1.0) < 0.25


def test_integer_inputs_are_small_integers():
    wl = synth.WORKLOADS["c4_scale_min"].resized(N=1, H=6, W=8)
    t = synth.make_integer_inputs(wl, seed=3)
    for v in (t.x, t.w, t.b):
        assert np.array_equal(v, np.round(v)) and np.all(np.abs(v) <= 8)
    # every product and partial sum stays an exact integer in fp32
    assert 9 * wl.Cin * 8 * 8 + 8 < 2 ** 24
