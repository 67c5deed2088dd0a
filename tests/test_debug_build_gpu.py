"""The device-checking build (libfa_gb300_debug.so, FA_DEBUG=1) on odd shapes.

Its prefill kernels check every TMA coordinate, every TMEM lane and column
range, and at the end of a launch every barrier's phase count, recording a
failure instead of trapping (include/fa.h, "Debug build"). This stands in for
a race and bounds checker: the odd-shaped cases below (ragged tails, Nq > Nk,
one query row, per-row and broadcast key masks, several units per CTA, e4m3
inputs) must leave the record clear and give outputs bit-identical to the
release library's, and a self-test shows that each check does fire on values
it must reject.
"""

import ctypes
import math

import pytest
import torch

from io_aware_exact_fa_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_fa_gb300 import build
    build.build()
    build.build(debug=True)
    from io_aware_exact_fa_gb300 import fa
    return fa, fa.lib, fa.debug_library()


def _record(lib):
    out = (ctypes.c_uint32 * 8)()
    assert lib.fa_debug_record(out, None) == 0
    return list(out)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _fwd(lib, q, k, v, scale, causal, words=None, strides=(0, 0, 0)):
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    if words is None:
        rc = lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, d,
                        ctypes.c_float(scale), int(causal), _stream())
    else:
        rc = lib.fa_fwd_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk,
                               d, ctypes.c_float(scale), int(causal), words.data_ptr(), *strides, _stream())
    assert rc == 0, lib.fa_last_error_detail()
    torch.cuda.synchronize()
    return o, lse


def _fwd8(lib, q8, k8, v8, ds, scale, causal):
    B, H, Nq, d = q8.shape
    Nk = k8.shape[2]
    o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    rc = lib.fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, d,
                        ctypes.c_float(scale), *(ctypes.c_float(x) for x in ds), int(causal), _stream())
    assert rc == 0, lib.fa_last_error_detail()
    torch.cuda.synchronize()
    return o, lse


def test_debug_build_flag_and_selftest(libs):
    fa, rel, dbg = libs
    assert dbg.fa_debug_enabled() == 1 and rel.fa_debug_enabled() == 0
    _record(dbg)                                   # start from a clear record
    assert dbg.fa_debug_selftest(None) == 0
    rec = _record(dbg)
    assert rec[0] == 1 | 2 | 4, rec               # TMA, TMEM and phase checks each fired
    assert rec[1] == 99 and rec[7] == 4, rec       # the self-test's site, four failed checks
    assert _record(dbg) == [0] * 8                 # reading the record cleared it
    assert rel.fa_debug_selftest(None) == 0        # the release build has no checks
    assert _record(rel) == [0] * 8
    assert dbg.fa_get_device_status(None) == 0


# B, H, Nq, Nk, d, causal, mask ("row": one row fully masked, "pad": a broadcast key mask)
CASES = [
    (1, 2, 1, 700, 64, False, None),
    (1, 3, 129, 513, 64, True, None),
    (2, 2, 513, 129, 128, True, None),          # Nq > Nk: early rows see no key
    (1, 2, 300, 257, 128, False, "row"),
    (2, 3, 384, 1000, 64, True, "pad"),          # broadcast key mask: one CTA per unit, trimmed key range
    (3, 64, 512, 512, 64, False, None),          # more units than SMs: several units per CTA
    (1, 48, 1000, 1000, 128, True, None),        # many causal units, longest first
]


@pytest.mark.parametrize("case", CASES, ids=[f"b{c[0]}h{c[1]}q{c[2]}k{c[3]}d{c[4]}{'c' if c[5] else ''}"
                                             f"{c[6] or ''}" for c in CASES])
def test_debug_build_clean_and_identical(libs, case):
    fa, rel, dbg = libs
    B, H, Nq, Nk, d, causal, mask = case
    q, k, v = (t.cuda() for t in W.make_qkv(B, H, Nq, Nk, d, seed=B * 1000 + Nq + Nk))
    words, strides = None, (0, 0, 0)
    if mask == "row":
        keep = torch.ones(B, H, Nq, Nk, dtype=torch.bool)
        keep[0, 1, 7] = False
        keep[:, :, :, 100:140] = False
        w = W.pack_keep_bits(keep)
        words, strides = w.cuda(), W.mask_strides(w)
    elif mask == "pad":
        w = W.pack_keep_bits(W.key_padding_keep(B, H, Nk, 2, 700))
        words, strides = w.cuda(), W.mask_strides(w)
    _record(dbg)
    scale = 1.0 / math.sqrt(d)
    o_d, l_d = _fwd(dbg, q, k, v, scale, causal, words, strides)
    rec = _record(dbg)
    assert rec == [0] * 8, f"debug checks failed: {rec}"
    assert dbg.fa_get_device_status(None) == 0
    o_r, l_r = _fwd(rel, q, k, v, scale, causal, words, strides)
    assert torch.equal(o_d, o_r) and torch.equal(l_d, l_r)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk,causal", [(200, 300, True), (513, 129, True), (1, 700, False)])
def test_debug_build_fp8_clean_and_identical(libs, Nq, Nk, causal, d):
    fa, rel, dbg = libs
    (q8, k8, v8), ds = W.make_qkv_fp8(2, 2, Nq, Nk, d, seed=Nq + Nk, device="cuda")
    _record(dbg)
    o_d, l_d = _fwd8(dbg, q8, k8, v8, ds, 1 / math.sqrt(d), causal)
    rec = _record(dbg)
    assert rec == [0] * 8, f"debug checks failed: {rec}"
    o_r, l_r = _fwd8(rel, q8, k8, v8, ds, 1 / math.sqrt(d), causal)
    assert torch.equal(o_d, o_r) and torch.equal(l_d, l_r)
