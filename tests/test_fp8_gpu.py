"""GPU parity of the FP8 forward pass (fa_fwd_fp8) against the fp64 oracle.

The oracle (oracle/fp8.py) is exact attention on the real values of the
e4m3 codes (code value times descale). The kernel computes the score and
value products on e4m3 operands with fp32 accumulation, which is exact for
the scores, and rounds P to e4m3 before the P V product. That rounding moves
a weight p by at most 2^-4 p (3 mantissa bits; below 2^-6 by at most 2^-10),
and the row sum l is taken before the rounding, so an output element moves
by at most 2^-4 max|v| plus the tiny-weight term. The tolerance is therefore
  max |dO| <= 2^-4 * max|v| + 1e-2 + half a bf16 ulp of the reference
  (1e-2 and the half ulp are the bf16 path's own bound),
  mean |dO| <= 4e-3   (the rounding errors of many weights cancel),
  |d lse| <= 1e-3     (lse uses l before the rounding: the bf16 path's bound),
and rows the oracle gives lse = -inf must return lse = -inf and O = 0.
"""

import math

import numpy as np
import pytest
import torch

from io_aware_exact_fa_gb300 import workloads as W
from oracle import fp8 as FP8
from tests.parity import half_ulp_bf16, to64

pytestmark = pytest.mark.gpu

TOL_MEAN = 4e-3
TOL_LSE = 1e-3


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_fa_gb300 import build
    build.build()
    from io_aware_exact_fa_gb300 import fa as lib
    return lib


def check(o, lse, ro, rl, vmax, what):
    """o, ro: [r, d]; lse, rl: [r]; vmax: max |v| of the head (real values)."""
    empty = np.isneginf(rl)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: -inf pattern of lse differs"
    assert np.all(o[empty] == 0), f"{what}: empty rows must be 0"
    d = np.abs(o - ro)
    bound = 2.0 ** -4 * vmax + 1e-2 + half_ulp_bf16(ro)
    assert np.all(d <= bound), f"{what}: max |dO| {d.max():.3e} over the bound (max bound {bound.max():.3e})"
    assert d.mean() <= TOL_MEAN, f"{what}: mean |dO| {d.mean():.3e}"
    fin = ~empty
    if fin.any():
        dl = np.abs(lse[fin] - rl[fin]).max()
        assert dl <= TOL_LSE, f"{what}: max |d lse| {dl:.3e}"
    return float(d.max()), float(d.mean())


def run(fa, q8, k8, v8, ds, scale, causal):
    o, lse = fa.fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), *ds, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    return to64(o), to64(lse)


CASES = [  # B, H, Nq, Nk, causal, scale
    (1, 2, 200, 300, False, None),
    (1, 2, 200, 300, True, None),
    (2, 1, 129, 513, False, None),
    (2, 1, 513, 129, True, None),     # Nq > Nk, bottom-right causal: early rows see no key
    (1, 1, 128, 128, True, None),
    (1, 3, 384, 384, False, -0.09),   # negative scale
    (1, 1, 1, 700, False, None),      # one query row
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", CASES, ids=[f"b{c[0]}h{c[1]}q{c[2]}k{c[3]}{'c' if c[4] else ''}"
                                             f"{'neg' if c[5] and c[5] < 0 else ''}" for c in CASES])
def test_fp8_parity_every_element(fa, case, d):
    B, H, Nq, Nk, causal, scale = case
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    (q8, k8, v8), ds = W.make_qkv_fp8(B, H, Nq, Nk, d, seed=Nq + 7 * Nk + H)
    o, lse = run(fa, q8, k8, v8, ds, scale, causal)
    stats = []
    for b in range(B):
        for h in range(H):
            ro, rl = FP8.attend_head_fp8(q8[b, h].numpy(), k8[b, h].numpy(), v8[b, h].numpy(), *ds, scale, causal)
            vmax = np.abs(FP8.dequantize(v8[b, h].numpy(), ds[2])).max()
            stats.append(check(o[b, h], lse[b, h], ro, rl, vmax, f"{case} b{b} h{h}"))
    print(case, "max/mean |dO|:", max(s[0] for s in stats), max(s[1] for s in stats))


def test_fp8_long_context_sampled(fa):
    """B=1 H=32 N=8192 d=128 causal (the long-context prefill workload) on
    e4m3 inputs: two whole heads and 256 seeded rows of four more heads."""
    B, H, N, d = 1, 32, 8192, 128
    scale = 1.0 / math.sqrt(d)
    (q8, k8, v8), ds = W.make_qkv_fp8(B, H, N, N, d, seed=0, device="cuda")
    o, lse = fa.fwd_fp8(q8, k8, v8, *ds, scale=scale, causal=True)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    rows = W.sample_rows(N, 256, seed=5).numpy()
    rows = np.unique(np.concatenate([rows, [0, N - 1]]))
    for h, rr in [(0, None), (31, None), (5, rows), (12, rows), (20, rows), (27, rows)]:
        qh, kh, vh = (t[0, h].cpu().numpy() for t in (q8, k8, v8))
        ro, rl = FP8.attend_head_fp8(qh, kh, vh, *ds, scale, True, rows=rr)
        sel = slice(None) if rr is None else rr
        vmax = np.abs(FP8.dequantize(vh, ds[2])).max()
        print(h, check(to64(o[0, h][sel]), to64(lse[0, h][sel]), ro, rl, vmax, f"8k head {h}"))


def test_fp8_headline_sampled(fa):
    """B=4 H=16 N=2048 d=64 (the headline prefill workload), both causal modes,
    on e4m3 inputs: three whole heads and 256 seeded rows of three more."""
    B, H, N, d = 4, 16, 2048, 64
    scale = 1.0 / math.sqrt(d)
    (q8, k8, v8), ds = W.make_qkv_fp8(B, H, N, N, d, seed=0, device="cuda")
    rows = np.unique(np.concatenate([W.sample_rows(N, 256, seed=11).numpy(), [0, N - 1]]))
    for causal in (False, True):
        o, lse = fa.fwd_fp8(q8, k8, v8, *ds, scale=scale, causal=causal)
        torch.cuda.synchronize()
        assert fa.device_status() == fa.FA_OK
        for (b, h), rr in [((0, 0), None), ((3, 15), None), ((2, 7), None), ((1, 3), rows), ((2, 9), rows),
                           ((3, 1), rows)]:
            qh, kh, vh = (t[b, h].cpu().numpy() for t in (q8, k8, v8))
            ro, rl = FP8.attend_head_fp8(qh, kh, vh, *ds, scale, causal, rows=rr)
            sel = slice(None) if rr is None else rr
            vmax = np.abs(FP8.dequantize(vh, ds[2])).max()
            check(to64(o[b, h][sel]), to64(lse[b, h][sel]), ro, rl, vmax, f"2k d64 causal={causal} ({b},{h})")


def test_fp8_deterministic(fa):
    for d in (64, 128):
        (q8, k8, v8), ds = W.make_qkv_fp8(2, 4, 1000, 1000, d, seed=9, device="cuda")
        a = fa.fwd_fp8(q8, k8, v8, *ds, causal=True)
        b = fa.fwd_fp8(q8, k8, v8, *ds, causal=True)
        torch.cuda.synchronize()
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fp8_rejects_bad_arguments(fa):
    q8 = torch.zeros(1, 1, 128, 96, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fwd_fp8(q8, q8, q8, 1.0, 1.0, 1.0)          # d = 96: not built
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    q8 = torch.zeros(1, 1, 128, 128, dtype=torch.uint8, device="cuda")
    for bad in ((0.0, 1.0, 1.0), (1.0, float("nan"), 1.0), (1.0, 1.0, -2.0)):
        with pytest.raises(fa.FAError) as e:
            fa.fwd_fp8(q8, q8, q8, *bad)
        assert e.value.status == fa.FA_ERR_INVALID_ARG
