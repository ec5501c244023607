"""Python binding of libconv_epi: fused 3x3 Conv2d + epilogue on GB300.

Argument marshalling only.  Every entry point has the name of the C function
it calls (include/conv_epi.h) and takes torch CUDA tensors (or, for
``conv_epi_forward_host``, numpy arrays / CPU tensors) in place of pointers.
Every step of the computation runs in the library's CUDA kernels; there is no
fallback: if ``libconv_epi.so`` is missing or the device is not sm_103a, the
calls raise.  Before a call, tensor arguments are checked for what their raw
addresses cannot carry: element type (float32, int32 for indices),
C-contiguity, and device or host memory as the call requires.  Their sizes
must match the problem description; plain integers pass as raw addresses.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libconv_epi.so")

MODE_TF32, MODE_FP32 = 0, 1
LAYOUT_NCHW, LAYOUT_NHWC = 0, 1
MIN_TANH2, SCALE_MIN, MUL_LRELU_GELU, GN_SCALE_POOL_CLAMP, NONE = 1, 2, 3, 4, 5
STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "ALIGNMENT", 4: "CUDA", 5: "TIMEOUT",
          6: "NO_MEMORY", 7: "DEVICE"}


class ConvEpiError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib().conv_epi_status_string(status).decode()
        if status == 4:
            msg += " -- " + _lib().conv_epi_last_cuda_error().decode()
        super().__init__(f"{where}: {STATUS.get(status, status)} ({msg})")


class Desc(C.Structure):
    _fields_ = [("N", C.c_int), ("Cin", C.c_int), ("H", C.c_int), ("W", C.c_int), ("Cout", C.c_int),
                ("mode", C.c_int),
                ("layout", C.c_int)]


class EpilogueDesc(C.Structure):
    _fields_ = [
        ("kind", C.c_int),
        ("scalar", C.c_float),
        ("chan_scale", C.c_void_p),
        ("lrelu_slope", C.c_float),
        ("groups", C.c_int),
        ("eps", C.c_float),
        ("gamma", C.c_void_p),
        ("beta", C.c_void_p),
        ("pool_k", C.c_int),
        ("clamp_lo", C.c_float),
        ("clamp_hi", C.c_float),
        ("index_out", C.c_void_p),
    ]


# conv_epi_plan (include/conv_epi.h), every field an int64_t, in declaration
# order; the library reports its own sizeof in struct_bytes, which
# conv_epi_plan_query checks against this layout
_PLAN_FIELDS = (
    "struct_bytes", "gemm_cout", "S", "P", "U", "RU", "Rin", "PL", "ucol", "chunks", "CT", "CW", "BW", "MT",
    "units_per_image", "resident", "na", "nb", "nr", "a_bytes", "b_bytes", "raw_bytes", "scratch_bytes",
    "a_off", "b_off", "raw_off", "bar_off", "scratch_off", "bar_bytes", "smem", "smem_limit",
    "a_plane_bytes", "a_lbo", "a_kw_stride", "x_pitch", "box[4]", "acc_cols", "tmem_cols", "conv_items",
    "wpack_bytes", "xpad_bytes", "gn_two_pass", "ybuf_bytes",
)


class Plan(C.Structure):
    _fields_ = [(f[:-3], C.c_int64 * 4) if f.endswith("[4]") else (f, C.c_int64) for f in _PLAN_FIELDS]


_lock = threading.Lock()
_L = None


def _lib():
    global _L
    with _lock:
        if _L is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build() "
                                   "(the CUDA path has no fallback)")
            L = C.CDLL(LIB_PATH)
            P, I = C.c_void_p, C.c_int
            L.conv_epi_status_string.restype = C.c_char_p
            L.conv_epi_status_string.argtypes = [I]
            L.conv_epi_last_cuda_error.restype = C.c_char_p
            L.conv_epi_output_shape.argtypes = [C.POINTER(Desc), C.POINTER(EpilogueDesc), P]
            L.conv_epi_create.argtypes = [C.POINTER(Desc), C.POINTER(P)]
            L.conv_epi_reserve.argtypes = [P, C.POINTER(EpilogueDesc)]
            L.conv_epi_forward.argtypes = [P, P, P, P, C.POINTER(EpilogueDesc), P, P]
            L.conv_epi_forward_host.argtypes = [P, P, P, P, C.POINTER(EpilogueDesc), P, P]
            L.conv_epi_forward_noalloc.argtypes = [C.POINTER(Desc), P, P, P, C.POINTER(EpilogueDesc), P, P]
            L.conv_epi_postpass.argtypes = [P, P, C.POINTER(EpilogueDesc), P, P]
            L.conv_epi_sync.argtypes = [P, P]
            L.conv_epi_noalloc_sync.argtypes = [P]
            L.conv_epi_test_drop_tile.argtypes = [P, I]
            L.conv_epi_plan_query.argtypes = [C.POINTER(Desc), C.POINTER(EpilogueDesc), C.POINTER(Plan)]
            L.conv_epi_destroy.argtypes = [P]
            L.conv_epi_workspace_bytes.argtypes = [P]
            L.conv_epi_workspace_bytes.restype = C.c_size_t
            L.conv_epi_last_launch_count.argtypes = [P]
            L.conv_epi_version.restype = I
            _L = L
    return _L


def _arg(t, what, device=None, index=False):
    """Address of a tensor argument after the checks a raw pointer cannot
    carry: element type (float32; int32 for an index output), C-contiguity
    and, where the call fixes it, device (True) or host (False) memory.
    None and plain integers (raw addresses) pass unchecked."""
    if t is None or isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):  # torch tensor
        import torch
        want = torch.int32 if index else torch.float32
        if t.dtype != want:
            raise TypeError(f"{what}: dtype {t.dtype}, expected {want}")
        if not t.is_contiguous():
            raise ValueError(f"{what}: not contiguous")
        if device is not None and bool(t.is_cuda) != device:
            raise ValueError(f"{what}: expected {'device' if device else 'host'} memory")
        return t.data_ptr()
    if hasattr(t, "ctypes"):  # numpy array: host memory
        import numpy as np
        want = np.int32 if index else np.float32
        if t.dtype != want:
            raise TypeError(f"{what}: dtype {t.dtype}, expected {np.dtype(want)}")
        if not t.flags.c_contiguous:
            raise ValueError(f"{what}: not C-contiguous")
        if device:
            raise ValueError(f"{what}: a numpy array is host memory; this call takes device memory")
        return t.ctypes.data
    return int(t)


def _tensors(x, w, b, epi, out, device):
    """The forward's pointer arguments, checked; the chain's tensors too."""
    keep = getattr(epi, "_keep", (None, None, None, None))
    for v, what, index in zip(keep, ("chan_scale", "gamma", "beta", "index_out"), (False, False, False, True)):
        _arg(v, what, device, index)
    return _arg(x, "x", device), _arg(w, "w", device), _arg(b, "b", device), _arg(out, "out", device)


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def _check(st, where):
    if st:
        raise ConvEpiError(st, where)


def epilogue(kind, scalar=1.0, chan_scale=None, lrelu_slope=0.01, groups=16, eps=1e-5, gamma=None, beta=None,
             pool_k=4, clamp_lo=0.0, clamp_hi=1.0, index_out=None):
    """Build a conv_epi_epilogue_desc; tensors are kept alive on the object."""
    e = EpilogueDesc(kind, scalar, _arg(chan_scale, "chan_scale"), lrelu_slope, groups, eps, _arg(gamma, "gamma"),
                     _arg(beta, "beta"), pool_k, clamp_lo, clamp_hi, _arg(index_out, "index_out", index=True))
    e._keep = (chan_scale, gamma, beta, index_out)
    return e


def conv_epi_output_shape(N, Cin, H, W, Cout, epi, mode=MODE_TF32, layout=LAYOUT_NCHW):
    import numpy as np
    s = np.zeros(4, dtype=np.int64)
    d = Desc(N, Cin, H, W, Cout, mode, layout)
    _check(_lib().conv_epi_output_shape(C.byref(d), C.byref(epi), s.ctypes.data), "conv_epi_output_shape")
    return tuple(int(v) for v in s)


def conv_epi_plan_query(N, Cin, H, W, Cout, epi, layout=LAYOUT_NCHW):
    """The tensor-core kernel's plan for this problem and chain (pure host
    call) as a dict; raises ConvEpiError where the kernel refuses the shape."""
    d = Desc(N, Cin, H, W, Cout, MODE_TF32, layout)
    q = Plan()
    _check(_lib().conv_epi_plan_query(C.byref(d), C.byref(epi), C.byref(q)), "conv_epi_plan_query")
    if q.struct_bytes != C.sizeof(Plan):
        raise RuntimeError(f"conv_epi_plan is {q.struct_bytes} bytes in the library, {C.sizeof(Plan)} here")
    return {name: (list(getattr(q, name)) if hasattr(getattr(q, name), "__len__") else int(getattr(q, name)))
            for name, _ in Plan._fields_}


def conv_epi_create(N, Cin, H, W, Cout, mode=MODE_TF32, layout=LAYOUT_NCHW):
    """layout: LAYOUT_NCHW (x[N][Cin][H][W]) or LAYOUT_NHWC (x[N][H][W][Cin];
    tf32 mode needs Cin a multiple of 4, fp32 mode takes any Cin)."""
    h = C.c_void_p()
    d = Desc(N, Cin, H, W, Cout, mode, layout)
    _check(_lib().conv_epi_create(C.byref(d), C.byref(h)), "conv_epi_create")
    return h


def conv_epi_reserve(h, epi):
    _check(_lib().conv_epi_reserve(h, C.byref(epi)), "conv_epi_reserve")


def conv_epi_forward(h, x, w, b, epi, out, stream=None):
    px, pw, pb, po = _tensors(x, w, b, epi, out, device=True)
    _check(_lib().conv_epi_forward(h, px, pw, pb, C.byref(epi), po, _stream(stream)), "conv_epi_forward")
    return out


def conv_epi_forward_host(h, x, w, b, epi, out, stream=None):
    px, pw, pb, po = _tensors(x, w, b, epi, out, device=False)
    _check(_lib().conv_epi_forward_host(h, px, pw, pb, C.byref(epi), po, _stream(stream)), "conv_epi_forward_host")
    return out


def conv_epi_forward_noalloc(N, Cin, H, W, Cout, x, w, b, epi, out, stream=None, mode=MODE_TF32,
                             layout=LAYOUT_NCHW):
    """Tensor-core forward without a handle: the library allocates nothing and
    uses its fixed device-side scratch array (see include/conv_epi.h)."""
    d = Desc(N, Cin, H, W, Cout, mode, layout)
    px, pw, pb, po = _tensors(x, w, b, epi, out, device=True)
    _check(_lib().conv_epi_forward_noalloc(C.byref(d), px, pw, pb, C.byref(epi), po, _stream(stream)),
           "conv_epi_forward_noalloc")
    return out


def conv_epi_postpass(h, y, epi, out, stream=None):
    """The chain alone over a stored conv output ``y`` [N, Cout, Ho, Wo]
    (device, float32, bias included), in fp32 arithmetic."""
    keep = getattr(epi, "_keep", (None, None, None, None))
    for v, what, index in zip(keep, ("chan_scale", "gamma", "beta", "index_out"), (False, False, False, True)):
        _arg(v, what, True, index)
    _check(_lib().conv_epi_postpass(h, _arg(y, "y", True), C.byref(epi), _arg(out, "out", True), _stream(stream)),
           "conv_epi_postpass")
    return out


def conv_epi_sync(h, stream=None):
    _check(_lib().conv_epi_sync(h, _stream(stream)), "conv_epi_sync")


def conv_epi_noalloc_sync(stream=None):
    """Wait for ``stream`` and raise if an allocation-free forward on the
    current device timed out since the last call (the error word is then
    cleared)."""
    _check(_lib().conv_epi_noalloc_sync(_stream(stream)), "conv_epi_noalloc_sync")


def conv_epi_test_drop_tile(h, tile):
    """Test hook: the next tf32 forward on ``h`` skips staged tile ``tile`` of
    every CTA's sequence, so its bounded waits time out (-1 cancels).  With
    ``h`` None it applies to the calling thread's next allocation-free
    forward."""
    _check(_lib().conv_epi_test_drop_tile(h, tile), "conv_epi_test_drop_tile")


def conv_epi_destroy(h):
    _check(_lib().conv_epi_destroy(h), "conv_epi_destroy")


def conv_epi_workspace_bytes(h):
    return _lib().conv_epi_workspace_bytes(h)


def conv_epi_last_launch_count(h):
    return _lib().conv_epi_last_launch_count(h)


def conv_epi_version():
    return _lib().conv_epi_version()


def conv_epi_status_string(status):
    return _lib().conv_epi_status_string(status).decode()


def conv_epi_last_cuda_error():
    """Text of the last failing CUDA call the library recorded."""
    return _lib().conv_epi_last_cuda_error().decode()


class ConvEpi:
    """Owns one handle; ``forward`` allocates the output with torch."""

    def __init__(self, N, Cin, H, W, Cout, mode=MODE_TF32, layout=LAYOUT_NCHW):
        self.dims = (N, Cin, H, W, Cout)
        self.mode = mode
        self.layout = layout
        self.h = conv_epi_create(N, Cin, H, W, Cout, mode, layout)

    def output_shape(self, epi):
        return conv_epi_output_shape(*self.dims, epi, self.mode, self.layout)

    def forward(self, x, w, b, epi, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty(self.output_shape(epi), device=x.device, dtype=torch.float32)
        return conv_epi_forward(self.h, x, w, b, epi, out, stream)

    def close(self):
        if self.h:
            conv_epi_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
