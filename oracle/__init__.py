"""fp64 CPU oracle for the fused 3x3 conv + epilogue chains (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  The
arithmetic lives in ``oracle.c`` (plain C, double precision); this file only
builds it with gcc and marshals numpy arrays.  It imports nothing from the
CUDA library's package.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

MIN_TANH2, SCALE_MIN, MUL_LRELU_GELU, GN_SCALE_POOL_CLAMP = 1, 2, 3, 4

_lock = threading.Lock()
_lib = None


class _Chain(C.Structure):
    _fields_ = [
        ("kind", C.c_int),
        ("scalar", C.c_double),
        ("mult", C.c_void_p),
        ("lrelu_slope", C.c_double),
        ("groups", C.c_int),
        ("eps", C.c_double),
        ("gamma", C.c_void_p),
        ("beta", C.c_void_p),
        ("scale", C.c_void_p),
        ("pool_k", C.c_int),
        ("clamp_lo", C.c_double),
        ("clamp_hi", C.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, -O2, no -march)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                               "-lpthread", "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            P = C.c_void_p
            I = C.c_int
            L.oracle_conv_out.argtypes = [I, I, C.POINTER(I), C.POINTER(I)]
            L.oracle_pool_out.argtypes = [I, I]
            L.oracle_pool_out.restype = I
            L.oracle_output_shape.argtypes = [I, I, I, I, I, C.POINTER(_Chain), P]
            L.oracle_conv3x3.argtypes = [P, P, P, I, I, I, I, I, P, I]
            L.oracle_chain_min.argtypes = [P, I, I, I, I, C.c_double, I, P, P]
            L.oracle_chain_mul_lrelu_gelu.argtypes = [P, I, I, I, I, P, C.c_double, P]
            L.oracle_chain_gn_pool.argtypes = [P, I, I, I, I, C.POINTER(_Chain), P, P, P, P]
            L.oracle_forward.argtypes = [P, P, P, I, I, I, I, I, C.POINTER(_Chain), P, P, I]
            L.oracle_conv_at.argtypes = [P, P, P, I, I, I, I, I, I, I, I, I]
            L.oracle_conv_at.restype = C.c_double
            L.oracle_min_at.argtypes = [P, P, P, I, I, I, I, I, C.c_double, I, I, P, P, P, P, P]
            L.oracle_mul_lrelu_gelu_at.argtypes = [P, P, P, I, I, I, I, I, P, C.c_double, I, P, P, P, P, P]
            L.oracle_gn_group.argtypes = [P, P, P, I, I, I, I, I, C.POINTER(_Chain), I, I, P, P, P, P, I]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def chain(kind, scalar=1.0, mult=None, lrelu_slope=0.01, groups=16, eps=1e-5, gamma=None,
          beta=None, scale=None, pool_k=4, clamp_lo=0.0, clamp_hi=1.0):
    """Chain descriptor; the numpy parameter arrays are kept alive on it."""
    keep = [_f32(mult), _f32(gamma), _f32(beta), _f32(scale)]
    c = _Chain(kind, scalar, _ptr(keep[0]), lrelu_slope, groups, eps, _ptr(keep[1]), _ptr(keep[2]),
               _ptr(keep[3]), pool_k, clamp_lo, clamp_hi)
    c._keep = keep
    return c


def chain_for(wl, t):
    """Chain descriptor of a synthetic workload (synth.Workload) and its tensors."""
    return chain(wl.kind, scalar=wl.scalar, mult=t.mult, lrelu_slope=wl.lrelu_slope, groups=wl.groups,
                 eps=wl.eps, gamma=t.gamma, beta=t.beta, scale=t.scale, pool_k=wl.pool_k,
                 clamp_lo=wl.clamp_lo, clamp_hi=wl.clamp_hi)


def conv_out(H, W):
    ho, wo = C.c_int(), C.c_int()
    if lib().oracle_conv_out(H, W, C.byref(ho), C.byref(wo)):
        raise ValueError("conv needs H, W >= 3")
    return ho.value, wo.value


def pool_out(Ho, k):
    return lib().oracle_pool_out(Ho, k)


def output_shape(N, Cin, H, W, Cout, ch):
    s = np.zeros(4, dtype=np.int64)
    if lib().oracle_output_shape(N, Cin, H, W, Cout, C.byref(ch), s.ctypes.data):
        raise ValueError("bad shape / chain")
    return tuple(int(v) for v in s)


def conv3x3(x, w, b, nthreads=None):
    x, w, b = _f32(x), _f32(w), _f32(b)
    N, Cin, H, W = x.shape
    Cout = w.shape[0]
    Ho, Wo = conv_out(H, W)
    y = np.empty((N, Cout, Ho, Wo), dtype=np.float64)
    if lib().oracle_conv3x3(_ptr(x), _ptr(w), _ptr(b), N, Cin, H, W, Cout, _ptr(y), _threads(nthreads)):
        raise ValueError("oracle_conv3x3 failed")
    return y


def chain_min(y, scalar=1.0, tanh2=True):
    y = np.ascontiguousarray(y, dtype=np.float64)
    N, Cc, Ho, Wo = y.shape
    out = np.empty((N, 1, Ho, Wo), dtype=np.float64)
    arg = np.empty((N, 1, Ho, Wo), dtype=np.int32)
    if lib().oracle_chain_min(_ptr(y), N, Cc, Ho, Wo, scalar, int(bool(tanh2)), _ptr(out), _ptr(arg)):
        raise ValueError("oracle_chain_min failed")
    return out, arg


def chain_mul_lrelu_gelu(y, mult, slope=0.01):
    y = np.ascontiguousarray(y, dtype=np.float64)
    mult = _f32(mult)
    out = np.empty_like(y)
    N, Cc, Ho, Wo = y.shape
    if lib().oracle_chain_mul_lrelu_gelu(_ptr(y), N, Cc, Ho, Wo, _ptr(mult), slope, _ptr(out)):
        raise ValueError("oracle_chain_mul_lrelu_gelu failed")
    return out


def chain_gn_pool(y, ch):
    y = np.ascontiguousarray(y, dtype=np.float64)
    N, Cc, Ho, Wo = y.shape
    Hp, Wp = pool_out(Ho, ch.pool_k), pool_out(Wo, ch.pool_k)
    out = np.empty((N, Cc, Hp, Wp), dtype=np.float64)
    arg = np.empty((N, Cc, Hp, Wp), dtype=np.int32)
    mean = np.empty((N, ch.groups), dtype=np.float64)
    rstd = np.empty((N, ch.groups), dtype=np.float64)
    if lib().oracle_chain_gn_pool(_ptr(y), N, Cc, Ho, Wo, C.byref(ch), _ptr(out), _ptr(arg), _ptr(mean),
                                  _ptr(rstd)):
        raise ValueError("oracle_chain_gn_pool failed")
    return out, arg, mean, rstd


def forward(x, w, b, ch, nthreads=None, want_index=True):
    """conv + chain, one image at a time; returns (out fp64, index int32 or None)."""
    x, w, b = _f32(x), _f32(w), _f32(b)
    N, Cin, H, W = x.shape
    Cout = w.shape[0]
    shape = output_shape(N, Cin, H, W, Cout, ch)
    out = np.empty(shape, dtype=np.float64)
    arg = np.empty(shape, dtype=np.int32) if want_index else None
    if lib().oracle_forward(_ptr(x), _ptr(w), _ptr(b), N, Cin, H, W, Cout, C.byref(ch), _ptr(out), _ptr(arg),
                            _threads(nthreads)):
        raise ValueError("oracle_forward failed")
    return out, arg


def conv_at(x, w, b, n, co, i, j):
    x, w, b = _f32(x), _f32(w), _f32(b)
    N, Cin, H, W = x.shape
    return lib().oracle_conv_at(_ptr(x), _ptr(w), _ptr(b), N, Cin, H, W, w.shape[0], n, co, i, j)


def min_at(x, w, b, n, i, j, scalar=1.0, tanh2=True):
    x, w, b = _f32(x), _f32(w), _f32(b)
    N, Cin, H, W = x.shape
    n, i, j = (np.ascontiguousarray(a, dtype=np.int32) for a in (n, i, j))
    out = np.empty(len(n), dtype=np.float64)
    arg = np.empty(len(n), dtype=np.int32)
    if lib().oracle_min_at(_ptr(x), _ptr(w), _ptr(b), N, Cin, H, W, w.shape[0], scalar, int(bool(tanh2)), len(n),
                           _ptr(n), _ptr(i), _ptr(j), _ptr(out), _ptr(arg)):
        raise ValueError("oracle_min_at failed")
    return out, arg


def mul_lrelu_gelu_at(x, w, b, mult, n, co, i, j, slope=0.01):
    x, w, b, mult = _f32(x), _f32(w), _f32(b), _f32(mult)
    N, Cin, H, W = x.shape
    n, co, i, j = (np.ascontiguousarray(a, dtype=np.int32) for a in (n, co, i, j))
    out = np.empty(len(n), dtype=np.float64)
    if lib().oracle_mul_lrelu_gelu_at(_ptr(x), _ptr(w), _ptr(b), N, Cin, H, W, w.shape[0], _ptr(mult), slope,
                                      len(n), _ptr(n), _ptr(co), _ptr(i), _ptr(j), _ptr(out)):
        raise ValueError("oracle_mul_lrelu_gelu_at failed")
    return out


def gn_group(x, w, b, ch, n, g, nthreads=None):
    """GN chain outputs of channels g*C/G .. of image n: (out [cpg,Hp,Wp], index, mean, rstd)."""
    x, w, b = _f32(x), _f32(w), _f32(b)
    N, Cin, H, W = x.shape
    Cout = w.shape[0]
    Ho, Wo = conv_out(H, W)
    cpg = Cout // ch.groups
    Hp, Wp = pool_out(Ho, ch.pool_k), pool_out(Wo, ch.pool_k)
    out = np.empty((cpg, Hp, Wp), dtype=np.float64)
    arg = np.empty((cpg, Hp, Wp), dtype=np.int32)
    mean, rstd = C.c_double(), C.c_double()
    if lib().oracle_gn_group(_ptr(x), _ptr(w), _ptr(b), N, Cin, H, W, Cout, C.byref(ch), n, g, _ptr(out),
                             _ptr(arg), C.addressof(mean), C.addressof(rstd), _threads(nthreads)):
        raise ValueError("oracle_gn_group failed")
    return out, arg, mean.value, rstd.value
