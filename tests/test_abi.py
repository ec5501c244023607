"""C-ABI checks that need no GPU: the library builds and loads, exports every
entry point the header declares, and its host-side validation answers
without touching a device."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import x3_conv2d_epilogue_gb300 as ce
from x3_conv2d_epilogue_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "conv_epi.h")


def exported_symbols():
    """Names the header declares as CONV_EPI_API entry points."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"CONV_EPI_API\s+[\w\s\*]*?\b(conv_epi_\w+)\s*\(", text)))


def header_plan_fields():
    """conv_epi_plan's int64_t fields in declaration order, read from the header."""
    with open(HEADER) as f:
        text = f.read()
    body = re.search(r"typedef struct \{((?:(?!typedef).)*?)\} conv_epi_plan;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    assert re.findall(r"(\w+)\s+[^;]+;", body) == ["int64_t"] * len(re.findall(r"[^;]+;", body))
    fields = []
    for decl in re.findall(r"int64_t\s+([^;]+);", body):
        for name in decl.split(","):
            m = re.fullmatch(r"\s*(\w+)\s*(?:\[(\d+)\])?\s*", name)
            fields.append((m.group(1), int(m.group(2)) if m.group(2) else 1))
    return fields


def test_binding_plan_matches_the_header():
    """The binding declares conv_epi_plan statically; its fields are the
    header's, in the same order and with the same array lengths."""
    got = [(n, getattr(t, "_length_", 1)) for n, t in ce.Plan._fields_]
    assert got == header_plan_fields()
    assert C.sizeof(ce.Plan) == 8 * sum(k for _, k in got)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ce.LIB_PATH):
        _build.build()
    return ce._lib()


def test_header_declares_the_api():
    names = exported_symbols()
    for must in ("conv_epi_create", "conv_epi_forward", "conv_epi_destroy", "conv_epi_forward_host",
                 "conv_epi_output_shape", "conv_epi_status_string", "conv_epi_sync"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in exported_symbols():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", ce.LIB_PATH], capture_output=True, text=True)
    if out.returncode:
        pytest.skip("nm not available")
    names = {ln.split()[-1] for ln in out.stdout.splitlines() if ln.strip()}
    assert names == set(exported_symbols())


def test_status_strings(lib):
    for s in range(8):
        assert ce.conv_epi_status_string(s)
    assert "unknown" in ce.conv_epi_status_string(99)
    assert ce.conv_epi_version() >= 10000


def shape(N, Cin, H, W, Cout, epi, mode=ce.MODE_TF32):
    return ce.conv_epi_output_shape(N, Cin, H, W, Cout, epi, mode)


def test_output_shapes(lib):
    assert shape(2, 16, 32, 32, 64, ce.epilogue(ce.MIN_TANH2)) == (2, 1, 30, 30)
    assert shape(128, 16, 256, 256, 64, ce.epilogue(ce.MIN_TANH2)) == (128, 1, 254, 254)
    assert shape(64, 64, 256, 256, 128, ce.epilogue(ce.SCALE_MIN, scalar=2.0)) == (64, 1, 254, 254)
    assert shape(64, 64, 256, 256, 64, ce.epilogue(ce.MUL_LRELU_GELU, chan_scale=16)) == (64, 64, 254, 254)
    gn = ce.epilogue(ce.GN_SCALE_POOL_CLAMP, chan_scale=16, gamma=16, beta=16, groups=16, pool_k=4)
    assert shape(128, 8, 128, 128, 64, gn) == (128, 64, 31, 31)


@pytest.mark.parametrize("bad", [
    dict(N=-1), dict(Cin=0), dict(H=2), dict(W=1), dict(Cout=0), dict(mode=7), dict(layout=2), dict(layout=-1),
])
def test_bad_descriptions_rejected(lib, bad):
    d = dict(N=1, Cin=4, H=8, W=8, Cout=8, mode=ce.MODE_FP32, layout=ce.LAYOUT_NCHW)
    d.update(bad)
    with pytest.raises(ce.ConvEpiError) as ei:
        ce.conv_epi_output_shape(d["N"], d["Cin"], d["H"], d["W"], d["Cout"], ce.epilogue(ce.MIN_TANH2), d["mode"],
                                 d["layout"])
    assert ei.value.status == 1


@pytest.mark.parametrize("mode,cin,want", [
    (ce.MODE_FP32, 6, 4),   # accepted, any Cin (the fp32 mode works on an NCHW copy): reaches the device
    (ce.MODE_TF32, 6, 2),   # a position's channels must start on 16-byte boundaries
    (ce.MODE_TF32, 8, 4),   # accepted: the call reaches the (absent) device
])
def test_channels_last_checked_before_the_device(lib, mode, cin, want):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = C.c_void_p()
    d = ce.Desc(1, cin, 8, 8, 8, mode, ce.LAYOUT_NHWC)
    assert lib.conv_epi_create(C.byref(d), C.byref(h)) == want and not h.value
    # the output shape does not depend on the input layout
    assert ce.conv_epi_output_shape(2, cin, 10, 12, 8, ce.epilogue(ce.MIN_TANH2), mode, ce.LAYOUT_NHWC) == (2, 1, 8, 10)


@pytest.mark.parametrize("kw", [
    dict(kind=9),
    dict(kind=ce.MUL_LRELU_GELU),                                     # no multiplier
    dict(kind=ce.MUL_LRELU_GELU, chan_scale=16, index_out=16),        # no index for this chain
    dict(kind=ce.GN_SCALE_POOL_CLAMP, chan_scale=16, gamma=16),       # no beta
    dict(kind=ce.GN_SCALE_POOL_CLAMP, chan_scale=16, gamma=16, beta=16, groups=3),   # 3 does not divide 8
    dict(kind=ce.GN_SCALE_POOL_CLAMP, chan_scale=16, gamma=16, beta=16, groups=2, pool_k=0),
    dict(kind=ce.GN_SCALE_POOL_CLAMP, chan_scale=16, gamma=16, beta=16, groups=2, pool_k=7),  # > Ho
    dict(kind=ce.GN_SCALE_POOL_CLAMP, chan_scale=16, gamma=16, beta=16, groups=2, clamp_lo=1, clamp_hi=0),
    dict(kind=ce.GN_SCALE_POOL_CLAMP, chan_scale=16, gamma=16, beta=16, groups=2, eps=-1.0),
    dict(kind=ce.SCALE_MIN, scalar=float("nan")),
])
def test_bad_chains_rejected(lib, kw):
    kind = kw.pop("kind")
    with pytest.raises(ce.ConvEpiError) as ei:
        ce.conv_epi_output_shape(1, 4, 8, 8, 8, ce.epilogue(kind, **kw))
    assert ei.value.status == 1


def test_null_pointers_rejected(lib):
    L = lib
    assert L.conv_epi_create(None, None) == 1
    assert L.conv_epi_forward(None, None, None, None, None, None, None) == 1
    assert L.conv_epi_forward_host(None, None, None, None, None, None, None) == 1
    assert L.conv_epi_destroy(None) == 1
    assert L.conv_epi_sync(None, None) == 1
    assert L.conv_epi_workspace_bytes(None) == 0
    assert L.conv_epi_output_shape(None, None, None) == 1
    assert L.conv_epi_test_drop_tile(None, -2) == 1
    # a null handle arms the hook for the calling thread's next allocation-free forward
    assert L.conv_epi_test_drop_tile(None, 0) == 0
    assert L.conv_epi_test_drop_tile(None, -1) == 0
    assert L.conv_epi_reserve(None, None) == 1
    assert L.conv_epi_forward_noalloc(None, None, None, None, None, None, None) == 1


def test_create_without_device_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = C.c_void_p()
    d = ce.Desc(1, 4, 8, 8, 8, ce.MODE_FP32)
    st = lib.conv_epi_create(C.byref(d), C.byref(h))
    assert st in (2, 4) and not h.value
    assert isinstance(ce.conv_epi_status_string(st), str)
    assert lib.conv_epi_noalloc_sync(None) == 4          # no device: a CUDA error, not a crash


def test_plain_conv_output_chain(lib):
    """CONV_EPI_NONE: the conv output itself, [N, Cout, Ho, Wo], no index
    output, in both modes."""
    e = ce.epilogue(ce.NONE)
    assert shape(2, 16, 32, 32, 64, e) == (2, 64, 30, 30)
    assert shape(3, 5, 9, 11, 200, e, ce.MODE_FP32) == (3, 200, 7, 9)
    with pytest.raises(ce.ConvEpiError) as ei:
        shape(1, 4, 8, 8, 8, ce.epilogue(ce.NONE, index_out=64))
    assert ei.value.status == 1
    q = ce.conv_epi_plan_query(64, 64, 256, 256, 64, e)     # planned like the per-channel chain
    r = ce.conv_epi_plan_query(64, 64, 256, 256, 64, ce.epilogue(ce.MUL_LRELU_GELU, chan_scale=16))
    assert q == r


def test_output_shapes_of_wide_and_many_channel_problems(lib):
    """Shapes the tf32 path runs in column and channel tiles have the plain
    output shapes (pure host call)."""
    shape = ce.conv_epi_output_shape
    assert shape(1, 16, 10, 520, 300, ce.epilogue(ce.MIN_TANH2)) == (1, 1, 8, 518)
    assert shape(2, 64, 7, 300, 200, ce.epilogue(ce.MUL_LRELU_GELU, chan_scale=16)) == (2, 200, 5, 298)
    gn = ce.epilogue(ce.GN_SCALE_POOL_CLAMP, chan_scale=16, gamma=16, beta=16, groups=16, pool_k=4)
    assert shape(3, 8, 18, 16, 64, gn) == (3, 64, 4, 3)


@pytest.mark.parametrize("layout,width,want", [
    (ce.LAYOUT_NCHW, 7, 4),    # accepted: rows of 7 floats are padded on the device
    (ce.LAYOUT_NHWC, 7, 4),    # accepted: channels-last rows need no padding
    (ce.LAYOUT_NCHW, 8, 4),
])
def test_tf32_takes_any_row_width(lib, layout, width, want):
    """Every W >= 3 reaches the device in tf32 mode (here: the absent one)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = C.c_void_p()
    d = ce.Desc(1, 8, 8, width, 64, ce.MODE_TF32, layout)
    assert lib.conv_epi_create(C.byref(d), C.byref(h)) == want and not h.value


def test_noalloc_refuses_rows_that_need_padding_before_the_device(lib):
    """The allocation-free forward has no buffer for the padded copy of NCHW
    rows whose width is not a multiple of 4: refused before any device call
    (the pointers are never dereferenced on the host)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    fake = C.c_void_p(1 << 20)  # 16-byte aligned, never touched
    epi = ce.epilogue(ce.SCALE_MIN)
    d = ce.Desc(1, 8, 8, 7, 64, ce.MODE_TF32, ce.LAYOUT_NCHW)
    assert lib.conv_epi_forward_noalloc(C.byref(d), fake, fake, fake, C.byref(epi), fake, None) == 2
    d = ce.Desc(1, 8, 8, 7, 64, ce.MODE_TF32, ce.LAYOUT_NHWC)  # channels last: reaches the device
    assert lib.conv_epi_forward_noalloc(C.byref(d), fake, fake, fake, C.byref(epi), fake, None) == 4


def test_binding_checks_tensor_arguments():
    """The binding refuses, before any library call, tensors whose element
    type, layout or memory a raw pointer cannot carry."""
    import torch
    f32 = torch.zeros(8)
    with pytest.raises(TypeError):
        ce.conv_epi_forward(None, torch.zeros(8, dtype=torch.float64), f32, f32, ce.epilogue(ce.SCALE_MIN), f32)
    with pytest.raises(ValueError):                                   # not contiguous
        ce.conv_epi_forward_host(None, torch.zeros(4, 4).t(), f32, f32, ce.epilogue(ce.SCALE_MIN), f32)
    with pytest.raises(ValueError):                                   # host tensor to a device call
        ce.conv_epi_forward(None, f32, f32, f32, ce.epilogue(ce.SCALE_MIN), f32)
    with pytest.raises(ValueError):                                   # numpy array to a device call
        ce.conv_epi_forward_noalloc(1, 8, 8, 8, 64, np.zeros(8, np.float32), f32, f32, ce.epilogue(ce.SCALE_MIN), f32)
    with pytest.raises(TypeError):                                    # the chain's parameters are float32
        ce.epilogue(ce.MUL_LRELU_GELU, chan_scale=np.zeros(8, np.float64))
    with pytest.raises(TypeError):                                    # indices are int32
        ce.epilogue(ce.SCALE_MIN, index_out=np.zeros(8, np.float32))
    with pytest.raises(ValueError):                                   # host parameters to a device call
        ce.conv_epi_forward(None, 1 << 20, 1 << 20, 1 << 20,
                            ce.epilogue(ce.MUL_LRELU_GELU, chan_scale=np.zeros(8, np.float32)), 1 << 20)


def test_empty_batch(lib):
    """N = 0 is a valid, empty problem: its output has no elements, and the
    allocation-free forward (which needs no handle) returns OK with null
    tensors and no device work, after the same chain checks and refusals."""
    assert ce.conv_epi_output_shape(0, 16, 10, 12, 64, ce.epilogue(ce.MIN_TANH2)) == (0, 1, 8, 10)
    gn = ce.epilogue(ce.GN_SCALE_POOL_CLAMP, chan_scale=16, gamma=16, beta=16, groups=16, pool_k=4)
    assert ce.conv_epi_output_shape(0, 8, 18, 16, 64, gn) == (0, 64, 4, 3)
    d = ce.Desc(0, 16, 10, 12, 64, ce.MODE_TF32, ce.LAYOUT_NCHW)
    assert lib.conv_epi_forward_noalloc(C.byref(d), None, None, None, C.byref(ce.epilogue(ce.MIN_TANH2)), None,
                                        None) == 0
    assert lib.conv_epi_forward_noalloc(C.byref(d), None, None, None, C.byref(ce.epilogue(9)), None, None) == 1
    assert lib.conv_epi_forward_noalloc(C.byref(d), None, None, None, C.byref(gn), None, None) == 2
    odd = ce.Desc(0, 16, 10, 13, 64, ce.MODE_TF32, ce.LAYOUT_NCHW)   # would need the padded copy
    assert lib.conv_epi_forward_noalloc(C.byref(odd), None, None, None, C.byref(ce.epilogue(ce.MIN_TANH2)), None,
                                        None) == 2
    full = ce.Desc(1, 16, 10, 12, 64, ce.MODE_TF32, ce.LAYOUT_NCHW)  # a non-empty batch still needs tensors
    assert lib.conv_epi_forward_noalloc(C.byref(full), None, None, None, C.byref(ce.epilogue(ce.MIN_TANH2)), None,
                                        None) == 1


def test_binding_has_every_entry_point():
    """The binding offers a function of the same name for every call the
    header declares."""
    assert [n for n in exported_symbols() if not callable(getattr(ce, n, None))] == []
    assert isinstance(ce.conv_epi_last_cuda_error(), str)


C_PROGRAM = r"""
#include <stdio.h>
#include "conv_epi.h"
int main(void) {
    conv_epi_desc d = {128, 16, 256, 256, 64, CONV_EPI_MODE_TF32, CONV_EPI_LAYOUT_NCHW};
    conv_epi_epilogue_desc e = {0};
    e.kind = CONV_EPI_MIN_TANH2;
    e.scalar = 1.0f;
    int64_t s[4];
    conv_epi_plan q;
    int st = (int)conv_epi_output_shape(&d, &e, s);
    int sq = (int)conv_epi_plan_query(&d, &e, &q);
    printf("%d %d %lld %lld %lld %lld %d %lld\n", conv_epi_version(), st, (long long)s[0], (long long)s[1],
           (long long)s[2], (long long)s[3], sq, (long long)q.struct_bytes);
    return 0;
}
"""


def test_plain_c_program_uses_the_abi(lib, tmp_path):
    """The header is plain C (C11, pedantic, no warnings) and a C program
    links against the library and calls it without any Python or torch."""
    import shutil
    import subprocess
    if not shutil.which("gcc"):
        pytest.skip("gcc not available")
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    pkg = os.path.dirname(ce.LIB_PATH)
    inc = os.path.dirname(HEADER)
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc, str(src), "-L", pkg,
                        "-lconv_epi", f"-Wl,-rpath,{pkg}", "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    assert int(out[0]) == ce.conv_epi_version()
    assert out[1:6] == ["0", "128", "1", "254", "254"]
    assert out[6] == "0" and int(out[7]) == ce.C.sizeof(ce.Plan)
