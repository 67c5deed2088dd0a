"""The C-ABI library builds for sm_103a, loads, and exports every symbol the
header declares; host-side argument checks fire before anything touches a
GPU (CPU only: no compute call is made here)."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    from io_aware_exact_fa_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def header_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", txt)))


def test_header_declares_the_api():
    names = header_functions()
    for need in ("fa_fwd", "fa_fwd_masked", "fa_decode_splitkv", "fa_decode_workspace_size",
                 "fa_get_device_status", "fa_status_string"):
        assert need in names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), f"{name} declared in fa.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", os.path.join(ROOT, "io_aware_exact_fa_gb300", "libfa_gb300.so")],
                         capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(fa_[a-z0-9_]+)$", out, flags=re.M))
    assert set(header_functions()) <= exported   # plain C names, not C++-mangled


def test_binding_covers_header():
    from io_aware_exact_fa_gb300 import fa
    assert set(header_functions()) == set(fa.EXPORTS)


def test_builds_for_sm103a_only():
    from io_aware_exact_fa_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    lib.fa_status_string.restype = ctypes.c_char_p
    assert lib.fa_status_string(0) == b"FA_OK"
    assert lib.fa_status_string(4) == b"FA_ERR_TIMEOUT"
    assert lib.fa_status_string(99) == b"FA_UNKNOWN_STATUS"


def test_workspace_size(lib):
    lib.fa_decode_workspace_size.restype = ctypes.c_size_t
    lib.fa_decode_workspace_size.argtypes = [ctypes.c_int] * 4
    n = lib.fa_decode_workspace_size(64, 32, 128, 16)
    parts = 64 * 32 * 16
    assert n >= parts * (128 + 2) * 4 and n % 256 == 0
    assert lib.fa_decode_workspace_size(1, 1, 96, 16) == 0
    assert lib.fa_decode_workspace_size(1, 1, 64, 0) == 0
    assert lib.fa_decode_workspace_size(0, 1, 64, 4) == 0


def _fwd(lib):
    f = lib.fa_fwd
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p]
    return f


def test_host_validation_before_launch(lib):
    """Invalid arguments are rejected on the host; no CUDA call is reached."""
    f = _fwd(lib)
    lib.fa_last_error_detail.restype = ctypes.c_char_p
    P = 1 << 20  # a fake, 16-byte aligned address that is never dereferenced
    assert f(None, P, P, P, None, 1, 1, 8, 8, 64, 0.125, 0, None) == 1          # NULL q
    assert f(P, P, P, P, None, 0, 1, 8, 8, 64, 0.125, 0, None) == 1             # B = 0
    assert f(P, P, P, P, None, 1, 1, -1, 8, 64, 0.125, 0, None) == 1            # Nq < 0
    assert f(P, P, P, P, None, 1, 1, 8, 0, 64, 0.125, 0, None) == 1             # Nk = 0
    assert f(P, P, P, P, None, 1, 1, 8, 8, 64, float("nan"), 0, None) == 1      # scale NaN
    assert f(P, P, P, P, None, 1, 1, 8, 8, 64, float("inf"), 0, None) == 1      # scale inf
    assert f(P, P, P, P, None, 1, 1, 8, 8, 96, 0.125, 0, None) == 2             # d = 96
    assert f(P + 8, P, P, P, None, 1, 1, 8, 8, 64, 0.125, 0, None) == 2         # misaligned q
    assert b"aligned" in lib.fa_last_error_detail()
    assert f(P, P, P, P, None, 1, 1, 0, 8, 64, 0.125, 0, None) == 0             # Nq = 0: no-op
    assert f(None, None, None, None, None, 1, 1, 0, 8, 64, 0.125, 0, None) == 0  # ... even with NULLs
    assert f(P, P, P, P, None, 1 << 16, 1 << 16, 8, 8, 64, 0.125, 0, None) == 1  # B*H too large


def test_decode_validation(lib):
    g = lib.fa_decode_splitkv
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p,
                                                                  ctypes.c_size_t, ctypes.c_void_p]
    P = 1 << 20
    big = 1 << 30
    assert g(None, P, P, P, None, 1, 1, 8, 64, 0.1, 4, P, big, None) == 1
    assert g(P, P, P, P, None, 1, 1, 8, 64, 0.1, 0, P, big, None) == 1          # no splits
    assert g(P, P, P, P, None, 1, 1, 8, 64, 0.1, 2000, P, big, None) == 1       # too many splits
    assert g(P, P, P, P, None, 1, 1, 8, 80, 0.1, 4, P, big, None) == 2          # d = 80
    assert g(P, P, P, P, None, 1, 1, 8, 64, 0.1, 4, None, big, None) == 5       # no workspace
    assert g(P, P, P, P, None, 1, 1, 8, 64, 0.1, 4, P, 16, None) == 5           # workspace too small
    assert g(P, P, P, P, None, 1, 1, 8, 64, 0.1, 4, P + 16, big, None) == 5     # workspace misaligned


def test_fwd_host_workspace_and_validation(lib):
    """The host-buffer forward pass: workspace size (two sets of q, k, v, o, lse
    per chunk of heads, each region rounded to 256 bytes) and the checks made
    before any CUDA call."""
    ws = lib.fa_fwd_host_workspace_size
    ws.restype = ctypes.c_size_t
    ws.argtypes = [ctypes.c_int] * 6
    up = lambda x: (x + 255) // 256 * 256
    # B=4 H=16 -> 64 heads, default chunk = 32 heads
    q, kv, lse = up(32 * 2048 * 64 * 2), up(32 * 2048 * 64 * 2), up(32 * 2048 * 4)
    assert ws(4, 16, 2048, 2048, 64, 0) == 2 * (2 * q + 2 * kv + lse)
    assert ws(4, 16, 2048, 2048, 64, 1000) == ws(4, 16, 2048, 2048, 64, 64)  # clamped to B*H
    assert ws(1, 3, 100, 300, 128, 2) == 2 * (2 * up(2 * 100 * 256) + 2 * up(2 * 300 * 256) + up(2 * 100 * 4))
    assert ws(1, 1, 8, 8, 96, 0) == 0 and ws(0, 1, 8, 8, 64, 0) == 0 and ws(1, 1, 8, 0, 64, 0) == 0
    f = lib.fa_fwd_host
    f.restype = ctypes.c_int
    f.argtypes = ([ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                                                ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p])
    P, big = 1 << 20, 1 << 30
    assert f(None, P, P, P, None, 1, 1, 8, 8, 64, 0.125, 0, 0, P, big, None) == 1       # NULL q
    assert f(P, P, P, P, None, 1, 1, 8, 8, 64, float("nan"), 0, 0, P, big, None) == 1   # scale NaN
    assert f(P, P, P, P, None, 1, 1, 8, 8, 80, 0.125, 0, 0, P, big, None) == 2          # d = 80
    assert f(P, P, P, P, None, 1, 1, 8, 8, 64, 0.125, 0, 0, None, big, None) == 5       # no workspace
    assert f(P, P, P, P, None, 1, 1, 8, 8, 64, 0.125, 0, 0, P, 64, None) == 5           # too small
    assert f(P, P, P, P, None, 1, 1, 8, 8, 64, 0.125, 0, 0, P + 16, big, None) == 5     # misaligned
    assert f(None, None, None, None, None, 1, 1, 0, 8, 64, 0.125, 0, 0, None, 0, None) == 0  # Nq = 0


def test_wait_limit_roundtrip(lib):
    lib.fa_get_wait_limit_ns.restype = ctypes.c_uint64
    lib.fa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    old = lib.fa_get_wait_limit_ns()
    lib.fa_set_wait_limit_ns(12345)
    assert lib.fa_get_wait_limit_ns() == 12345
    lib.fa_set_wait_limit_ns(old)
