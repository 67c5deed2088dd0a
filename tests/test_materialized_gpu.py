"""GPU parity of the materialising baseline (fa_fwd_materialized).

S = scale Q K^T goes through HBM in bf16 and so does P, so this path is less
precise than the fused kernel. Its tolerance is derived from that rounding:
every score moves by at most eps = 2^-9 max|s| (half a bf16 ulp, relative), so
lse moves by at most eps and each weight by a factor within e^(+-2 eps) after
normalisation, which moves O by at most (e^(2 eps) - 1) max|v|; rounding P
(relative 2^-9) adds up to 2^-8 max|v|, and the bf16 output half an ulp.
"""

import math

import numpy as np
import pytest
import torch

from io_aware_exact_fa_gb300 import workloads as W
from oracle import attention as A
from parity import half_ulp_bf16, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_fa_gb300 import build
    build.build()
    from io_aware_exact_fa_gb300 import fa as lib
    return lib


def bounds(q, k, v, scale):
    q64, k64, v64 = to64(q), to64(k), to64(v)
    smax = max(np.abs(scale * np.einsum("bhid,bhjd->bhij", q64, k64)).max(), 1e-30)
    eps = 2.0 ** -9 * smax
    vmax = np.abs(v64).max()
    return (math.exp(2 * eps) - 1) * vmax + 2.0 ** -8 * vmax + 1e-3, eps + 1e-3


def check(o, lse, o_ref, lse_ref, tol_o, tol_l, what):
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), what
    assert np.all(o[empty] == 0), what
    excess = np.abs(o - o_ref) - half_ulp_bf16(o_ref)
    assert excess.max() <= tol_o, f"{what}: {excess.max():.3e} > {tol_o:.3e}"
    dl = np.abs(lse[~empty] - lse_ref[~empty]).max(initial=0.0)
    assert dl <= tol_l, f"{what}: lse {dl:.3e} > {tol_l:.3e}"
    return float(excess.max()), float(dl)


@pytest.mark.parametrize("d", [64, 128])
# rows of up to ~7k keys take the warp-per-row softmax; Nk = 8192 the CTA-per-row one
@pytest.mark.parametrize("shape", [(1, 2, 200, 256), (2, 1, 300, 264), (1, 1, 129, 520), (1, 2, 520, 128),
                                   (1, 1, 70, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_materialized_vs_oracle(fa, shape, d):
    B, H, Nq, Nk = shape
    q, k, v = W.make_qkv(B, H, Nq, Nk, d, seed=Nq + Nk + d)
    scale = 1.0 / math.sqrt(d)
    tol_o, tol_l = bounds(q, k, v, scale)
    for causal in (False, True):
        o, lse = fa.fwd_materialized(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal)
        torch.cuda.synchronize()
        o_ref = np.zeros((B, H, Nq, d))
        lse_ref = np.zeros((B, H, Nq))
        for b in range(B):
            for h in range(H):
                o_ref[b, h], lse_ref[b, h] = A.attend_head(to64(q[b, h]), to64(k[b, h]), to64(v[b, h]), scale, causal)
        print(shape, d, causal, check(to64(o), to64(lse), o_ref, lse_ref, tol_o, tol_l, f"{shape} d={d} {causal}"))


def test_materialized_matches_fused(fa):
    """The bench workload: the baseline and the fused kernel compute the same attention."""
    w = W.WORKLOADS["prefill_2k"]
    q, k, v = W.make_qkv(1, 4, w.Nq, w.Nk, w.d, seed=0)
    tol_o, tol_l = bounds(q, k, v, w.scale)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    for causal in (False, True):
        om, lm = fa.fwd_materialized(qc, kc, vc, scale=w.scale, causal=causal)
        of, lf = fa.fwd(qc, kc, vc, scale=w.scale, causal=causal)
        torch.cuda.synchronize()
        # the fused result is within 1e-2 (+ half an ulp) of the exact one
        check(to64(om), to64(lm), to64(of), to64(lf), tol_o + 1e-2, tol_l + 1e-3, f"vs fused causal={causal}")


def test_materialized_rejects(fa):
    x = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(1, 1, 12, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:   # Nk = 12 is not a multiple of 8
        fa.fwd_materialized(x, y, y)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    with pytest.raises(fa.FAError) as e:
        fa.fwd_materialized(x, x, x, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == fa.FA_ERR_WORKSPACE
