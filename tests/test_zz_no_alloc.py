"""Split-KV decode through the allocation-free entry point.

fa_decode_splitkv_noalloc serves callers that cannot allocate device memory
(they hold only their input and output buffers): it keeps the per-split
partial states in the library's static device scratch. Its results must
match the regular entry point, which uses a caller workspace, on two calls
in a row (the second call reuses the scratch the first one left behind).
This file is collected last on purpose.
"""

import ctypes
import math

import pytest
import torch

from io_aware_exact_fa_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_fa_gb300 import build
    build.build()
    from io_aware_exact_fa_gb300 import fa
    return fa


def _noalloc(fa, q, k, v, o, lse, scale, splits):
    f = fa.lib.fa_decode_splitkv_noalloc          # the C ABI directly
    B, H, _, d = q.shape
    return f(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, k.shape[2], d,
             ctypes.c_float(scale), splits, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_twice(lib):
    fa = lib
    for (B, H, Nk, d, S, seed) in [(8, 32, 8192, 128, 16, 0), (3, 5, 777, 64, 7, 1)]:
        q, k, v = W.make_qkv(B, H, 1, Nk, d, seed=seed, device="cuda")
        scale = 1.0 / math.sqrt(d)
        ref_o, ref_l = fa.decode(q, k, v, scale=scale, num_splits=S)
        torch.cuda.synchronize()
        for call in range(2):
            o = torch.full_like(q, float("nan"))
            lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
            assert _noalloc(fa, q, k, v, o, lse, scale, S) == fa.FA_OK, fa.lib.fa_last_error_detail()
            torch.cuda.synchronize()
            assert fa.device_status() == fa.FA_OK
            # the same kernels on the same bytes: the outputs must be bit-identical
            assert torch.equal(o, ref_o), f"noalloc call {call + 1} {(B, H, Nk, d, S)}: o differs"
            assert torch.equal(lse, ref_l), f"noalloc call {call + 1} {(B, H, Nk, d, S)}: lse differs"


def test_noalloc_rejects_requests_beyond_the_static_scratch(lib):
    fa = lib
    B, H, d, S = 64, 64, 128, 16          # 64*64*16 partials * (128 + 2) * 4 B > 20 MiB
    assert fa.decode_workspace_size(B, H, d, S) > fa.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(B, H, 1, d, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(B, H, 1, d, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, H, dtype=torch.float32, device="cuda")
    assert _noalloc(fa, q, kv, kv, o, lse, 0.1, S) == fa.FA_ERR_WORKSPACE
    assert b"static scratch" in fa.lib.fa_last_error_detail()
