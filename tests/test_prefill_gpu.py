"""GPU parity of the fused prefill kernel against the fp64 oracle (same bytes).

Small cases compare every output element; the full-size workloads compare
whole heads plus seeded samples of rows from every head.
"""

import math

import numpy as np
import pytest
import torch

from io_aware_exact_fa_gb300 import workloads as W
from tests.parity import compare, oracle_heads, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_fa_gb300 import build
    build.build()
    from io_aware_exact_fa_gb300 import fa as lib
    return lib


def run(fa, q, k, v, scale, causal, keep=None):
    """Copy CPU bf16 inputs to the GPU, run through the C ABI, return CPU fp64 (O, lse)."""
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    kb, strides = None, (0, 0, 0)
    if keep is not None:
        words = W.pack_keep_bits(keep)
        strides = W.mask_strides(words)
        kb = words.cuda()
    o, lse = fa.fwd(dq, dk, dv, scale=scale, causal=causal, keep_bits=kb, mask_strides=strides)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    return to64(o), to64(lse)


def check_full(fa, q, k, v, scale, causal, keep=None, what=""):
    o, lse = run(fa, q, k, v, scale, causal, keep)
    ref = oracle_heads(q, k, v, scale, causal, keep)
    B, H = q.shape[:2]
    ro = np.stack([np.stack([ref[(b, h)][0] for h in range(H)]) for b in range(B)])
    rl = np.stack([np.stack([ref[(b, h)][1] for h in range(H)]) for b in range(B)])
    return compare(o, lse, ro, rl, what)


# --------------------------------------------------------------- 128 x 128 case
@pytest.mark.parametrize("causal", [False, True])
def test_pr1_offsets_and_masked_row(fa, causal):
    """1 head, 128 x 128, d 64, scale 1/8; rows 124-127 shifted by +/-1e3 through Q,
    row 64 fully key-masked (expected O = 0, lse = -inf)."""
    w = W.WORKLOADS["pr1"]
    q, k, v = W.make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, seed=0)
    q, k = W.add_row_offsets(q, k, w.scale)
    keep = W.pr1_keep()
    st = check_full(fa, q, k, v, w.scale, causal, keep, f"pr1 causal={causal}")
    o, lse = run(fa, q, k, v, w.scale, causal, keep)
    assert np.all(o[0, 0, W.PR1_MASKED_ROW] == 0) and np.isneginf(lse[0, 0, W.PR1_MASKED_ROW])
    for r, s in zip(W.PR1_OFFSET_ROWS, W.PR1_OFFSET_SIGNS):
        assert abs(lse[0, 0, r] - s * 1e3) < 60, "offset rows carry a ~1e3 lse"
    print(st)


def test_pr1_no_mask_both_modes(fa):
    w = W.WORKLOADS["pr1"]
    q, k, v = W.make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, seed=0)
    for causal in (False, True):
        check_full(fa, q, k, v, w.scale, causal, None, f"pr1 plain causal={causal}")


def test_shift_invariance_on_gpu(fa):
    """Adding a row constant c to every score leaves O unchanged and moves lse by c."""
    q, k, v = W.make_qkv(1, 2, 256, 384, 128, seed=3)
    k = k.clone()
    k[..., -1] = 1.0
    o0, l0 = run(fa, q, k, v, 1 / math.sqrt(128), False)
    for c in (1e3, -1e3):
        q2 = q.float().clone()
        q2[..., -1] += c * math.sqrt(128)
        q2 = q2.to(torch.bfloat16)
        shift = (q2.double()[..., -1] - q.double()[..., -1]) / math.sqrt(128)   # exact per-row constant
        o1, l1 = run(fa, q2, k, v, 1 / math.sqrt(128), False)
        assert np.abs(o1 - o0).max() < 1e-2
        assert np.abs((l1 - l0) - shift.numpy()).max() < 2e-3


def test_large_score_spread(fa):
    """Rows scaled so their scores span about +/-1e3 (most weights underflow)."""
    q, k, v = W.make_qkv(1, 1, 128, 256, 64, seed=4)
    q = W.scale_rows(q, [60.0, -60.0, 120.0], [5, 77, 127])
    for causal in (False, True):
        check_full(fa, q, k, v, 0.125, causal, None, f"spread causal={causal}")


# ------------------------------------------------------------- ragged shapes
SHAPES = [
    (1, 1, 1, 1), (1, 1, 1, 200), (1, 2, 100, 77), (2, 1, 300, 257), (1, 1, 129, 520),
    (1, 3, 513, 1000), (2, 2, 256, 256), (1, 1, 255, 129), (1, 1, 1000, 64),
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_ragged(fa, shape, d):
    B, H, Nq, Nk = shape
    q, k, v = W.make_qkv(B, H, Nq, Nk, d, seed=Nq * 7 + Nk)
    for causal in (False, True):
        check_full(fa, q, k, v, 1 / math.sqrt(d), causal, None, f"{shape} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_key_padding_and_row_masks(fa, d):
    g = torch.Generator().manual_seed(9)
    q, k, v = W.make_qkv(2, 3, 300, 450, d, seed=5)
    # key padding, broadcast over rows
    kp = torch.ones(2, 3, 1, 450, dtype=torch.bool)
    kp[0, 1, 0, 200:] = False      # trailing keys padded: later key tiles are skipped
    kp[1, 2, 0, :130] = False      # leading keys masked
    kp[0, 2, 0, :] = False         # a head with no key at all: O = 0, lse = -inf
    for causal in (False, True):
        check_full(fa, q, k, v, 0.1, causal, kp, f"keypad causal={causal}")
    # an arbitrary per-row mask, with some fully masked rows
    keep = torch.rand(2, 3, 300, 450, generator=g) < 0.3
    keep[0, 0, 17] = False
    keep[1, 1, 299] = False
    for causal in (False, True):
        check_full(fa, q, k, v, 0.1, causal, keep, f"rowmask causal={causal}")


# ------------------------------------------- several units per persistent CTA
@pytest.mark.parametrize("d", [64, 128])
def test_many_units_per_cta(fa, d):
    """B*H*ceil(Nq/256) well above the SM count, so every persistent CTA walks
    several units with barrier phases running on across them. Nq = 300 leaves
    the second Q tile of each head's last pair empty (rows from 384), and under
    the causal mask the first tiles visit 1-3 key tiles, so units of different
    lengths (and a first tile longer than the second) follow each other."""
    q, k, v = W.make_qkv(4, 48, 300, 300, d, seed=21)
    for causal in (False, True):
        check_full(fa, q, k, v, 1 / math.sqrt(d), causal, None, f"many units d={d} causal={causal}")
    keep = torch.rand(4, 48, 300, 300, generator=torch.Generator().manual_seed(4)) < 0.5
    check_full(fa, q, k, v, 1 / math.sqrt(d), True, keep, f"many units row mask d={d}")


@pytest.mark.parametrize("d", [64, 128])
def test_many_units_repeated(fa, d):
    """Barrier phases that run on across units must stay in step on every run:
    30 launches of a shape whose units alternate between two busy tiles and one
    tile with no key tiles (B=4, H=48, Nq=Nk=300) must all finish without a
    timed-out wait and give bit-identical outputs."""
    q, k, v = W.make_qkv(4, 48, 300, 300, d, seed=23)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    for causal in (False, True):
        ref = fa.fwd(dq, dk, dv, causal=causal)
        for _ in range(30):
            o, lse = fa.fwd(dq, dk, dv, causal=causal)
            assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1])
        torch.cuda.synchronize()
        assert fa.device_status() == fa.FA_OK


@pytest.mark.parametrize("d", [64, 128])
def test_many_units_rectangular(fa, d):
    """Nq != Nk with several units per CTA: 480 units of 6 key tiles each
    (non-causal), and bottom-right causal alignment with Nk > Nq."""
    q, k, v = W.make_qkv(2, 80, 520, 700, d, seed=22)
    for causal in (False, True):
        check_full(fa, q, k, v, 1 / math.sqrt(d), causal, None, f"rect units d={d} causal={causal}")


def test_scale_zero_is_uniform(fa):
    q, k, v = W.make_qkv(1, 1, 130, 140, 64, seed=6)
    check_full(fa, q, k, v, 0.0, False, None, "scale 0")
    keep = torch.rand(1, 1, 130, 140, generator=torch.Generator().manual_seed(2)) < 0.5
    check_full(fa, q, k, v, 0.0, True, keep, "scale 0 masked causal")


def test_deterministic(fa):
    q, k, v = W.make_qkv(2, 4, 640, 640, 128, seed=8)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    a = fa.fwd(dq, dk, dv, causal=True)
    b = fa.fwd(dq, dk, dv, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_lse_optional_and_nq_zero(fa):
    q, k, v = W.make_qkv(1, 2, 200, 300, 64, seed=10)
    o1, _ = fa.fwd(q.cuda(), k.cuda(), v.cuda(), with_lse=False)
    o2, _ = fa.fwd(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    z = torch.empty(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    o, lse = fa.fwd(z, k.cuda(), v.cuda())
    assert o.shape == (1, 2, 0, 64)


def test_rejects_unsupported(fa):
    q = torch.zeros(1, 1, 8, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fwd(q, q, q)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    with pytest.raises(fa.FAError) as e:
        x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
        fa.fwd(x, x, x, scale=float("nan"))
    assert e.value.status == fa.FA_ERR_INVALID_ARG


def test_bounded_wait_reports_timeout_and_context_survives(fa):
    assert fa.selftest_wait_timeout(2_000_000) == fa.FA_ERR_TIMEOUT   # 2 ms limit
    assert fa.device_status() == fa.FA_OK                               # cleared
    q, k, v = W.make_qkv(1, 1, 128, 128, 64, seed=0)
    check_full(fa, q, k, v, 0.125, True, None, "after timeout self-test")


# ------------------------------------------------------- full-size workloads
def _sampled(fa, w, causal, keep=None, full_heads=2, rows_per_head=256, seed=0):
    """Every row of the first and last head (full_heads=2), plus rows_per_head
    seeded rows (and the first and last row) of every head."""
    q, k, v = W.make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, seed=seed)
    o, lse = run(fa, q, k, v, w.scale, causal, keep)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    full = heads[:1] + heads[-1:] if full_heads >= 2 else heads[:full_heads]
    ref = oracle_heads(q, k, v, w.scale, causal, keep, heads=full)
    for (b, h) in full:
        compare(o[b, h], lse[b, h], ref[(b, h)][0], ref[(b, h)][1], f"{w.name} head {b},{h}")
    rows = W.sample_rows(w.Nq, rows_per_head, seed=1).numpy()
    rows = np.unique(np.concatenate([rows, [0, w.Nq - 1]]))
    ref = oracle_heads(q, k, v, w.scale, causal, keep, rows=rows)
    go = np.stack([o[b, h][rows] for b, h in heads])
    gl = np.stack([lse[b, h][rows] for b, h in heads])
    ro = np.stack([ref[bh][0] for bh in heads])
    rl = np.stack([ref[bh][1] for bh in heads])
    return compare(go, gl, ro, rl, f"{w.name} sampled rows")


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_2k_d64(fa, causal):
    w = W.WORKLOADS["prefill_2k"]
    print(_sampled(fa, w, causal, full_heads=2, rows_per_head=128))


@pytest.mark.slow
def test_prefill_8k_d128_causal(fa):
    w = W.WORKLOADS["prefill_8k"]
    print(_sampled(fa, w, True, full_heads=2, rows_per_head=1024))


@pytest.mark.slow
def test_prefill_32k_d128_causal(fa):
    w = W.WORKLOADS["prefill_32k"]
    print(_sampled(fa, w, True, full_heads=2, rows_per_head=1024))


@pytest.mark.slow
def test_prefill_32k_d128_causal_keypad(fa):
    w = W.WORKLOADS["prefill_32k_pad"]
    keep = W.key_padding_keep(w.B, w.H, w.Nk, w.pad_heads, w.pad_from)
    print(_sampled(fa, w, True, keep=keep, full_heads=2, rows_per_head=1024))


def test_fma_pipe_exp2_error_bound(fa):
    """The FMA-pipe exponential stays within its stated 7.5e-5 relative error of 2^x."""
    x = torch.cat([torch.linspace(-125.0, 127.0, 1_000_001), torch.tensor([0.0, -0.5, 0.5, 8.0, -20.25])])
    y = fa.selftest_exp2(x.cuda()).cpu().double()
    ref = torch.exp2(x.double())
    rel = ((y - ref).abs() / ref).max().item()
    assert rel < 8e-5, rel
    # below the clamp (x < -125) the result stays at about 2^-125, negligible next
    # to the row maximum's 2^0
    y2 = fa.selftest_exp2(torch.tensor([-126.0, -200.0, -1000.0], device="cuda")).cpu().double()
    assert torch.all(y2 <= 2.0 ** -124) and torch.all(y2 > 0)
