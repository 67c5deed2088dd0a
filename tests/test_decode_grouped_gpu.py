"""GPU parity of the decode variants (fa_decode_grouped) against the fp64 oracle.

Grouped K/V heads (G = H / Hkv query heads per K/V head), Nq new tokens per
sequence with the causal rule among them, and per-sequence KV lengths,
including lengths of 0, lengths below Nq (tokens that see no key), lengths
that are not multiples of the 128-key tile, and more splits than key tiles.
Tolerances are those of the forward pass (tests/parity.py).
"""

import math

import numpy as np
import pytest
import torch

from io_aware_exact_fa_gb300 import workloads as W
from oracle import decode_variants as DV
from parity import compare, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_fa_gb300 import build
    build.build()
    from io_aware_exact_fa_gb300 import fa as lib
    return lib


def _inputs(B, H, Hkv, Nq, Nk, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, Nk, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, Nk, d, generator=g).to(torch.bfloat16)
    return q, k, v


def _run(fa, q, k, v, lens, splits, scale):
    sl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse = fa.decode_grouped(q.cuda(), k.cuda(), v.cuda(), seqlens_k=sl, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    return to64(o), to64(lse)


# B, H, Hkv, Nq, Nk, lens, splits
CASES = [
    (2, 4, 4, 1, 300, None, 1),                # one head per K/V head, one token
    (2, 8, 2, 1, 1000, [1000, 517], 3),        # G = 4
    (3, 8, 1, 2, 700, [0, 1, 700], 2),         # G = 8; lengths 0 and below Nq
    (2, 16, 4, 4, 2000, [129, 1999], 4),       # G = 4, 4 new tokens
    (1, 32, 2, 8, 640, [640], 5),              # G = 16, 8 tokens: 128 rows per tile
    (2, 4, 2, 3, 130, [2, 130], 7),            # more splits than key tiles
    (2, 6, 3, 5, 257, [5, 256], 1),            # one split over several tiles, Nq = L for one sequence
    (2, 4, 2, 1, 777, [777, 65], 3),           # G = 2: two rows per K/V head
    (3, 6, 2, 1, 500, [0, 1, 500], 2),         # G = 3: three rows (a padded row), lengths 0 and 1
    (2, 8, 4, 2, 900, [1, 899], 4),            # G = 2, 2 tokens: four rows; a length below Nq
    (1, 2, 2, 3, 250, [250], 2),               # G = 1, 3 tokens
    (2, 5, 1, 1, 400, [400, 130], 2),          # G = 5: one row past the CUDA-core kernel's four
    (1, 17, 1, 1, 300, [300], 2),              # G = 17: one row past the keys-on-lanes kernel's sixteen
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}kv{}nq{}nk{}s{}".format(*c[:5], c[6]))
def test_decode_grouped(fa, case, d):
    B, H, Hkv, Nq, Nk, lens, splits = case
    q, k, v = _inputs(B, H, Hkv, Nq, Nk, d, seed=B * 1000 + H * 10 + Nq)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, q, k, v, lens, splits, scale)
    o_ref, lse_ref = DV.decode_grouped_attention(to64(q), to64(k), to64(v), lens, scale)
    st = compare(o.reshape(-1, d), lse.reshape(-1), o_ref.reshape(-1, d), lse_ref.reshape(-1),
                 f"{case} d={d}")
    print(case, d, st)


@pytest.mark.parametrize("d,Nq", [(64, 1), (64, 4), (128, 1)])
def test_decode_grouped_deterministic(fa, d, Nq):
    """Each split kernel (the CUDA-core kernel at d = 64 with one token, the
    keys-on-lanes kernel otherwise) and the merge sum in a fixed order: two
    calls on the same inputs give identical bytes."""
    q, k, v = _inputs(2, 8, 2, Nq, 1500, d, seed=11)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    lens = torch.tensor([1500, 777], dtype=torch.int32, device="cuda")
    o1, l1 = fa.decode_grouped(q, k, v, seqlens_k=lens, num_splits=3)
    o2, l2 = fa.decode_grouped(q, k, v, seqlens_k=lens, num_splits=3)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_grouped_matches_splitkv_layout(fa):
    """G = 1, Nq = 1, no lengths: the same attention as fa_decode_splitkv (both
    against the oracle, and against each other within twice the tolerance)."""
    q, k, v = _inputs(4, 8, 8, 1, 1500, 128, seed=5)
    o_g, l_g = _run(fa, q, k, v, None, 6, 1 / math.sqrt(128))
    o_s, l_s = fa.decode(q.cuda(), k.cuda(), v.cuda(), num_splits=6)
    torch.cuda.synchronize()
    assert np.abs(o_g - to64(o_s)).max() <= 2e-2
    assert np.abs(l_g.reshape(-1) - to64(l_s).reshape(-1)).max() <= 2e-3


@pytest.mark.parametrize("Nq,d", [(2, 64), (1, 64), (1, 128)])
def test_decode_grouped_offsets(fa, Nq, d):
    """Rows whose scores sit near +/-1e3 (through a constant last key component):
    the reference max handling must keep them finite and exact."""
    B, H, Hkv, Nk = 1, 8, 2, 700
    q, k, v = _inputs(B, H, Hkv, Nq, Nk, d, seed=77)
    scale = 1.0 / 8.0
    k = k.clone()
    k[..., -1] = 1.0
    qf = q.float()
    qf[0, 1, 0, -1] += 1e3 / scale
    qf[0, 6, Nq - 1, -1] -= 1e3 / scale
    q = qf.to(torch.bfloat16)
    lens = [650]
    o, lse = _run(fa, q, k, v, lens, 3, scale)
    o_ref, lse_ref = DV.decode_grouped_attention(to64(q), to64(k), to64(v), lens, scale)
    compare(o.reshape(-1, d), lse.reshape(-1), o_ref.reshape(-1, d), lse_ref.reshape(-1), "offsets")


@pytest.mark.parametrize("name", ["gqa", "gqa_spec", "gqa_d64", "gqa_spec_d64"])
def test_decode_grouped_full_size_sampled(fa, name):
    """The benchmark's workloads and inputs (seed 0): 48 seeded (b, h) heads, all tokens."""
    w = W.DECODE_VARIANTS[name]
    q, k, v, lens = W.make_decode_inputs(w, seed=0)
    o, lse = fa.decode_grouped(q.cuda(), k.cuda(), v.cuda(), seqlens_k=lens.cuda(), scale=w.scale,
                               num_splits=w.num_splits)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    gen = torch.Generator().manual_seed(3)
    idx = torch.randperm(w.B * w.H, generator=gen)[:46].tolist() + [0, w.B * w.H - 1]
    heads = [(i // w.H, i % w.H) for i in idx]
    o_ref, lse_ref = DV.decode_grouped_attention(q, k, v, lens.tolist(), w.scale, heads=heads)
    og, lg = to64(o), to64(lse)
    sel = np.array(heads)
    compare(og[sel[:, 0], sel[:, 1]].reshape(-1, w.d), lg[sel[:, 0], sel[:, 1]].reshape(-1),
            o_ref[sel[:, 0], sel[:, 1]].reshape(-1, w.d), lse_ref[sel[:, 0], sel[:, 1]].reshape(-1), name)


def test_decode_grouped_rejects(fa):
    q = torch.zeros(1, 6, 1, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 4, 128, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:   # H not a multiple of Hkv
        fa.decode_grouped(q, k, k)
    assert e.value.status == fa.FA_ERR_INVALID_ARG
    q = torch.zeros(1, 32, 5, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:   # 32 * 5 = 160 query rows per K/V head
        fa.decode_grouped(q, k, k)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    q = torch.zeros(1, 2, 1, 96, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 1, 128, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.decode_grouped(q, k, k)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    q = torch.zeros(1, 2, 1, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.decode_grouped(q, k, k, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == fa.FA_ERR_WORKSPACE
