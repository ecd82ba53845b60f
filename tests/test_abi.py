"""The C ABI boundary, checked without a GPU.

The library must build for sm_103a, load, and export every entry point that
include/fa.h declares; the ctypes binding must match each declaration's
parameter list; argument validation that precedes any device work must return
the documented error codes.
"""
import ctypes
import os
import re

import pytest

from exact_io_aware_flash_gb300 import _lib, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fa.h")

C_TO_CTYPES = {
    "int": ctypes.c_int, "float": ctypes.c_float, "size_t": ctypes.c_size_t,
}


def declarations():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    decls = {}
    for m in re.finditer(r"FA_API\s+([\w\s\*]+?)\s*\b(fa_\w+)\s*\(([^)]*)\)\s*;", text, flags=re.S):
        ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
        plist = [] if params in ("", "void") else [p.strip() for p in params.split(",")]
        decls[name] = (ret, plist)
    return decls


def _ctype_of(param: str):
    p = " ".join(param.replace("const", "").split())
    if "*" in p:
        return ctypes.c_void_p if not p.startswith("char") else ctypes.c_char_p
    typ = p.split()[0]
    return C_TO_CTYPES[typ]


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_header_declares_the_boundary():
    d = declarations()
    for name in ("fa_forward", "fa_backward", "fa_backward_workspace_size", "fa_check_errors",
                 "fa_last_error", "fa_version"):
        assert name in d, name


def test_library_exports_every_declared_symbol(lib):
    for name in declarations():
        assert hasattr(lib, name), f"libfa.so does not export {name}"


def test_binding_signatures_match_header(lib):
    for name, (ret, params) in declarations().items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, name
        assert len(fn.argtypes) == len(params), f"{name}: {len(fn.argtypes)} vs {len(params)}"
        for got, p in zip(fn.argtypes, params):
            want = _ctype_of(p)
            if want is ctypes.c_void_p:
                assert got in (ctypes.c_void_p,), (name, p, got)
            else:
                assert got is want, (name, p, got)


def test_version_and_workspace_size(lib):
    assert "sm_103a" in _lib.version()
    B, Hq, N, d = 2, 3, 1000, 128
    rows = B * Hq * N
    assert _lib.workspace_size(B, Hq, N, d) == ((rows * 4 + 255) // 256) * 256
    assert _lib.workspace_size(0, 1, 1, 64) == 0


def test_invalid_arguments_fail_before_device_work(lib):
    fake = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    null = ctypes.c_void_p(0)
    # null pointer
    assert lib.fa_forward(null, fake, fake, fake, fake, 1, 1, 1, 8, 64, 0, 1.0, 0, null) == 1
    # Hq not a multiple of Hkv
    assert lib.fa_forward(fake, fake, fake, fake, fake, 1, 3, 2, 8, 64, 0, 1.0, 0, null) == 1
    # non-finite scale
    assert lib.fa_forward(fake, fake, fake, fake, fake, 1, 1, 1, 8, 64, 0, float("nan"), 0, null) == 1
    # unsupported head dimension and dtype
    assert lib.fa_forward(fake, fake, fake, fake, fake, 1, 1, 1, 8, 96, 0, 1.0, 0, null) == 2
    assert lib.fa_forward(fake, fake, fake, fake, fake, 1, 1, 1, 8, 64, 0, 1.0, 7, null) == 2
    # misaligned pointer
    odd = ctypes.c_void_p(4096 + 2)
    assert lib.fa_forward(odd, fake, fake, fake, fake, 1, 1, 1, 8, 64, 0, 1.0, 0, null) == 2
    assert b"aligned" in lib.fa_last_error()
    # workspace too small
    assert lib.fa_backward(fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, 16,
                           1, 1, 1, 8, 64, 0, 1.0, 0, null) == 1
    assert b"workspace" in lib.fa_last_error()


def test_window_entry_points_validate_before_device_work(lib):
    fake = ctypes.c_void_p(4096)
    null = ctypes.c_void_p(0)
    # window must be at least 1
    assert lib.fa_forward_window(fake, fake, fake, fake, fake, 1, 1, 1, 8, 64, 0, 1.0, 0, null) == 1
    assert b"window" in lib.fa_last_error()
    assert lib.fa_forward_window(fake, fake, fake, fake, fake, 1, 1, 1, 8, 64, -3, 1.0, 0, null) == 1
    # the checks shared with fa_forward still apply
    assert lib.fa_forward_window(null, fake, fake, fake, fake, 1, 1, 1, 8, 64, 4, 1.0, 0, null) == 1
    assert lib.fa_forward_window(fake, fake, fake, fake, fake, 1, 1, 1, 8, 96, 4, 1.0, 0, null) == 2
    assert lib.fa_backward_window(fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, 1 << 20,
                                  1, 1, 1, 8, 64, 0, 1.0, 0, null) == 1
    assert lib.fa_backward_window(fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, 16,
                                  1, 1, 1, 8, 64, 4, 1.0, 0, null) == 1
    assert b"workspace" in lib.fa_last_error()


def test_fp8_entry_points_validate_before_device_work(lib):
    fake = ctypes.c_void_p(4096)
    null = ctypes.c_void_p(0)
    assert lib.fa_fp8_vt_stride(1) == 16 and lib.fa_fp8_vt_stride(300) == 304
    assert lib.fa_fp8_vt_stride(0) == 0 and lib.fa_fp8_vt_stride(2 ** 31 - 1) == 0
    # d must be 128
    assert lib.fa_quantize_fp8(fake, fake, fake, null, fake, fake, fake, fake, fake, fake,
                               1, 1, 1, 8, 64, 1, null) == 2
    assert lib.fa_forward_fp8(fake, fake, fake, fake, fake, fake, fake, fake, 1, 1, 1, 8, 64, 0, 1.0,
                              null) == 2
    # null tensor, GQA divisibility
    assert lib.fa_quantize_fp8(null, fake, fake, null, fake, fake, fake, fake, fake, fake,
                               1, 1, 1, 8, 128, 1, null) == 1
    assert lib.fa_forward_fp8(fake, fake, fake, fake, fake, fake, fake, fake, 1, 3, 2, 8, 128, 0, 1.0,
                              null) == 1
