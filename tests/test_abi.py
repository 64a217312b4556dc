"""The C-ABI library builds, loads and exports every entry point its header
declares; host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

from paged_kv_decode_ns_gb300 import _build

HEADER = os.path.join(_build.INCLUDE, "ns_paged.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)      # drop comments
    text = re.sub(r"//[^\n]*", "", text)
    return sorted(set(re.findall(r"\b(ns_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    path = _build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_hot_path():
    names = _declared()
    for want in ("ns_kv_append", "ns_paged_attn_decode", "ns_paged_attn_prefill",
                 "ns_kv_append_paged_attn_decode", "ns_paged_attn_workspace_bytes"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_library_has_no_torch_dependency():
    import subprocess
    out = subprocess.run(["ldd", _build.LIB], capture_output=True, text=True).stdout
    assert "torch" not in out and "c10" not in out


def test_status_strings_and_version(lib):
    lib.ns_status_string.restype = ctypes.c_char_p
    for code in (0, -1, -2, -3, -4):
        assert lib.ns_status_string(code).startswith(b"NS_")
    assert lib.ns_version() >= 100


def test_host_checks_need_no_gpu(lib):
    P = ctypes.c_void_p
    f = lib.ns_kv_append
    f.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int64, ctypes.c_int, P]
    # null pointers
    assert f(None, None, None, None, None, 4, 2, 64, 16, 10, 0, None) == -1
    # unsupported head_dim / block_size / dtype
    assert f(None, None, None, None, None, 4, 2, 96, 16, 10, 0, None) == -2
    assert f(None, None, None, None, None, 4, 2, 128, 8, 10, 0, None) == -2
    # head_dim 128 with block_size 16 passes the shape checks
    assert f(None, None, None, None, None, 4, 2, 128, 16, 10, 0, None) == -1
    assert f(None, None, None, None, None, 4, 2, 64, 12, 10, 0, None) == -2
    assert f(None, None, None, None, None, 4, 2, 64, 16, 10, 7, None) == -2
    # zero tokens is a no-op
    assert f(None, None, None, None, None, 0, 2, 64, 16, 10, 0, None) == 0

    d = lib.ns_paged_attn_decode
    d.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_float, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                  P, ctypes.c_size_t]
    # 14 q heads over 4 kv heads is not a grouping
    assert d(None, None, None, None, None, 4, 14, 4, 64, 16, 0.125, None, None, 8, 10, 0, None, 0) == -2
    # 9 q heads per kv head: more than 8, and not cut evenly into groups of at most 8
    assert d(None, None, None, None, None, 4, 18, 2, 64, 16, 0.125, None, None, 8, 10, 0, None, 0) == -2
    # more than 64 q heads per kv head
    assert d(None, None, None, None, None, 4, 72, 1, 64, 16, 0.125, None, None, 8, 10, 0, None, 0) == -2
    # 16 q heads per kv head (two groups of 8) passes the shape checks
    assert d(None, None, None, None, None, 4, 32, 2, 64, 16, 0.125, None, None, 8, 10, 0, None, 0) == -1
    # null pointers
    assert d(None, None, None, None, None, 4, 14, 2, 64, 16, 0.125, None, None, 8, 10, 0, None, 0) == -1


def test_workspace_size_grows_with_rows(lib):
    w = lib.ns_paged_attn_workspace_bytes
    w.restype = ctypes.c_size_t
    w.argtypes = [ctypes.c_int] * 4
    a, b = w(1, 14, 2, 64), w(100000, 14, 2, 64)
    assert 0 < a < b
    assert b - a >= 99999 * 2 * 4          # at least one counter per (row, kv head)
    assert w(-1, 14, 2, 64) == 0
