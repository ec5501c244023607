"""Seeded synthetic inputs for the fused 3x3 conv + epilogue workloads.

This module is shared by the oracle tests, the CUDA parity tests, ``bench.py``
and ``__graft_entry__.smoke()``.  It holds no arithmetic of the method itself:
only a counter-based random generator, the five workload recipes and helpers
that draw their tensors.

Generator
---------
SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; Vigna's reference C code): the k-th output of a
stream whose state starts at ``s`` is ``mix(s + (k + 1) * 0x9E3779B97F4A7C15)``
with ``mix(z) = z1 ^ (z1 >> 31)``, ``z1 = (z0 ^ (z0 >> 27)) * 0x94D049BB133111EB``,
``z0 = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9`` (all mod 2**64).  Because the
k-th draw depends only on ``k``, any element of any tensor can be regenerated on
its own, which the sampled full-size checks use.

* uniform in [0, 1): top 53 bits of a draw times 2**-53;
* normal: Box-Muller, ``sqrt(-2 ln(1 - u1)) * cos(2 pi u2)`` with ``u1, u2``
  the draws at counters ``2k`` and ``2k + 1`` of the tensor's stream;
* every tensor has its own stream, keyed by ``(seed, stream id)``; the ids are
  fixed below in the order x, w, b, extra parameters.

All tensors are returned as contiguous float32 NCHW numpy arrays.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20

# stream ids, in the fixed draw order x, w, b, then the chain's parameters
STREAM_X, STREAM_W, STREAM_B, STREAM_MULT, STREAM_GAMMA, STREAM_BETA, STREAM_SCALE = range(7)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_state(seed: int, stream: int) -> np.uint64:
    """Initial SplitMix64 state of stream ``stream`` under ``seed``."""
    with np.errstate(over="ignore"):
        s = np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        s = _mix(s + np.uint64(stream + 1) * _GAMMA)
    return s[0]


def splitmix64(state: np.uint64, counters: np.ndarray) -> np.ndarray:
    """Draws number ``counters`` (uint64 array) of the stream starting at ``state``."""
    with np.errstate(over="ignore"):
        return _mix(state + (counters.astype(np.uint64) + np.uint64(1)) * _GAMMA)


def uniform01(state: np.uint64, counters: np.ndarray) -> np.ndarray:
    return (splitmix64(state, counters) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _fill(n: int, fn) -> np.ndarray:
    """Evaluate ``fn(counters)`` over ``0..n-1`` in chunks, on a thread pool
    (numpy's ufuncs release the GIL, so the chunks run in parallel)."""
    out = np.empty(n, dtype=np.float32)

    def one(lo):
        hi = min(n, lo + _CHUNK)
        out[lo:hi] = fn(np.arange(lo, hi, dtype=np.uint64))

    starts = range(0, n, _CHUNK)
    if n <= _CHUNK:
        for lo in starts:
            one(lo)
    else:
        with ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
            list(ex.map(one, starts))
    return out


def uniform(shape, lo: float, hi: float, seed: int, stream: int) -> np.ndarray:
    st = stream_state(seed, stream)
    n = int(np.prod(shape))
    return _fill(n, lambda k: lo + (hi - lo) * uniform01(st, k)).reshape(shape)


def normal(shape, mean: float, std: float, seed: int, stream: int) -> np.ndarray:
    st = stream_state(seed, stream)
    n = int(np.prod(shape))

    def draw(k):
        u1 = uniform01(st, 2 * k)
        u2 = uniform01(st, 2 * k + np.uint64(1))
        return mean + std * np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * math.pi * u2)

    return _fill(n, draw).reshape(shape)


def normal_at(flat_index: np.ndarray, mean: float, std: float, seed: int, stream: int) -> np.ndarray:
    """Elements ``flat_index`` of the tensor ``normal(...)`` would draw, on their own."""
    st = stream_state(seed, stream)
    k = np.asarray(flat_index, dtype=np.uint64)
    u1 = uniform01(st, 2 * k)
    u2 = uniform01(st, 2 * k + np.uint64(1))
    return (mean + std * np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * math.pi * u2)).astype(np.float32)


# ---------------------------------------------------------------------------
# workload recipes
# ---------------------------------------------------------------------------
KIND_MIN_TANH2 = 1
KIND_SCALE_MIN = 2
KIND_MUL_LRELU_GELU = 3
KIND_GN_SCALE_POOL_CLAMP = 4
KIND_NONE = 5  # the conv output itself, no chain


@dataclass(frozen=True)
class Workload:
    name: str
    N: int
    Cin: int
    H: int
    W: int
    Cout: int
    kind: int
    scalar: float = 1.0
    lrelu_slope: float = 0.01
    groups: int = 16
    eps: float = 1e-5
    pool_k: int = 4
    clamp_lo: float = 0.0
    clamp_hi: float = 1.0
    desc: str = field(default="", compare=False)

    def with_batch(self, n: int) -> "Workload":
        d = self.__dict__.copy()
        d["N"] = n
        return Workload(**d)

    def resized(self, **kw) -> "Workload":
        d = self.__dict__.copy()
        d.update(kw)
        return Workload(**d)


# The five workloads: shapes, chains and parameter distributions as stated for
# the pages' four models (tiny check case + four full-size cases).
WORKLOADS = {
    "pr1_min_tanh2": Workload("pr1_min_tanh2", 2, 16, 32, 32, 64, KIND_MIN_TANH2,
                              desc="x[2,16,32,32] conv 16->64, min over C, tanh, tanh"),
    "c2_min_tanh2": Workload("c2_min_tanh2", 128, 16, 256, 256, 64, KIND_MIN_TANH2,
                             desc="x[128,16,256,256] conv 16->64, min over C, tanh, tanh"),
    "c3_mul_lrelu_gelu": Workload("c3_mul_lrelu_gelu", 64, 64, 256, 256, 64, KIND_MUL_LRELU_GELU,
                                  desc="x[64,64,256,256] conv 64->64, x mult[C], LeakyReLU 0.01, erf GELU"),
    "c4_scale_min": Workload("c4_scale_min", 64, 64, 256, 256, 128, KIND_SCALE_MIN, scalar=2.0,
                             desc="x[64,64,256,256] conv 64->128, x 2.0, min over C"),
    "c5_gn_pool_clamp": Workload("c5_gn_pool_clamp", 128, 8, 128, 128, 64, KIND_GN_SCALE_POOL_CLAMP,
                                 desc="x[128,8,128,128] conv 8->64, GroupNorm 16, x scale[C], MaxPool 4, clamp [0,1]"),
}


@dataclass
class Tensors:
    x: np.ndarray
    w: np.ndarray
    b: np.ndarray
    mult: np.ndarray | None = None   # per-channel multiplier (E-full chain)
    gamma: np.ndarray | None = None  # GroupNorm weight
    beta: np.ndarray | None = None   # GroupNorm bias
    scale: np.ndarray | None = None  # per-channel scale after GroupNorm


def make_inputs(wl: Workload, seed: int = 0, x_scale: float = 1.0) -> Tensors:
    """Draw the workload's tensors: x ~ N(0,1); w, b ~ U(+-1/sqrt(Cin*9));
    multiplier ~ N(0,1); GroupNorm gamma ~ N(1,0.1), beta ~ N(0,0.1);
    scale ~ N(1,0.5)."""
    bound = 1.0 / math.sqrt(wl.Cin * 9)
    x = normal((wl.N, wl.Cin, wl.H, wl.W), 0.0, x_scale, seed, STREAM_X)
    w = uniform((wl.Cout, wl.Cin, 3, 3), -bound, bound, seed, STREAM_W)
    b = uniform((wl.Cout,), -bound, bound, seed, STREAM_B)
    t = Tensors(x, w, b)
    if wl.kind == KIND_MUL_LRELU_GELU:
        t.mult = normal((wl.Cout,), 0.0, 1.0, seed, STREAM_MULT)
    if wl.kind == KIND_GN_SCALE_POOL_CLAMP:
        t.gamma = normal((wl.Cout,), 1.0, 0.1, seed, STREAM_GAMMA)
        t.beta = normal((wl.Cout,), 0.0, 0.1, seed, STREAM_BETA)
        t.scale = normal((wl.Cout,), 1.0, 0.5, seed, STREAM_SCALE)
    return t


def make_integer_inputs(wl: Workload, seed: int = 0, amp: int = 8) -> Tensors:
    """Integer-valued x, w, b in [-amp, amp]: every product and partial sum of
    the conv is an integer below 2**24, so fp32 and tf32 hold them exactly."""
    def ints(shape, stream):
        st = stream_state(seed, stream)
        n = int(np.prod(shape))
        return _fill(n, lambda k: (splitmix64(st, k) % np.uint64(2 * amp + 1)).astype(np.float64) - amp).reshape(shape)
    x = ints((wl.N, wl.Cin, wl.H, wl.W), STREAM_X)
    w = ints((wl.Cout, wl.Cin, 3, 3), STREAM_W)
    b = ints((wl.Cout,), STREAM_B)
    t = Tensors(x, w, b)
    if wl.kind == KIND_MUL_LRELU_GELU:
        t.mult = normal((wl.Cout,), 0.0, 1.0, seed, STREAM_MULT)
    if wl.kind == KIND_GN_SCALE_POOL_CLAMP:
        t.gamma = normal((wl.Cout,), 1.0, 0.1, seed, STREAM_GAMMA)
        t.beta = normal((wl.Cout,), 0.0, 0.1, seed, STREAM_BETA)
        t.scale = normal((wl.Cout,), 1.0, 0.5, seed, STREAM_SCALE)
    return t
