"""GPU parity of the backward pass (fa_bwd) against the fp64 backward oracle.

The CUDA path recomputes P from the lse its own forward pass wrote and rounds
P and dS to bf16 for the tensor-core products; the oracle uses the exact P.
Each gradient is compared relative to its own scale: max |d| / max |ref| and
mean |d| / mean |ref| (a gradient is a sum over up to N terms, so an absolute
bound would depend on N).
"""

import math

import numpy as np
import pytest
import torch

from io_aware_exact_fa_gb300 import workloads as W
from oracle import attention_grad as AG

pytestmark = pytest.mark.gpu

TOL_MAX_REL = 2e-2
TOL_MEAN_REL = 1e-2


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_fa_gb300 import build
    build.build()
    from io_aware_exact_fa_gb300 import fa as lib
    return lib


def make_dout(B, H, Nq, d, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16)


def gpu_grads(fa, q, k, v, do, scale, causal):
    dq_, dk_, dv_, do_ = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.fwd(dq_, dk_, dv_, scale=scale, causal=causal)
    gq, gk, gv = fa.bwd(dq_, dk_, dv_, o, lse, do_, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    return [t.double().cpu().numpy() for t in (gq, gk, gv)]


def compare_grads(got, ref, what):
    stats = {}
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.all(np.isfinite(g)), f"{what} {name}: non-finite"
        d = np.abs(g - r)
        scale_max, scale_mean = np.abs(r).max(), np.abs(r).mean()
        if scale_max == 0:
            assert d.max() == 0, f"{what} {name}: expected exact zeros"
            continue
        mx, mean = d.max() / scale_max, d.mean() / scale_mean
        stats[name] = (float(mx), float(mean))
        assert mx <= TOL_MAX_REL, f"{what} {name}: max rel {mx:.3e}"
        assert mean <= TOL_MEAN_REL, f"{what} {name}: mean rel {mean:.3e}"
    return stats


SHAPES = [(1, 1, 128, 128), (1, 2, 200, 200), (2, 1, 300, 257), (1, 1, 129, 520), (1, 2, 513, 300)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_backward_ragged(fa, shape, d):
    B, H, Nq, Nk = shape
    q, k, v = W.make_qkv(B, H, Nq, Nk, d, seed=Nq + 3 * Nk)
    do = make_dout(B, H, Nq, d, seed=Nq * 5 + Nk)
    scale = 1 / math.sqrt(d)
    for causal in (False, True):
        got = gpu_grads(fa, q, k, v, do, scale, causal)
        ref = AG.attention_grad(q, k, v, do, scale, causal)
        print(shape, d, causal, compare_grads(got, ref, f"{shape} d={d} causal={causal}"))


def test_backward_rectangular_causal(fa):
    """Bottom-right causal with Nq != Nk: with Nq > Nk the first Nq - Nk queries
    see no key (their dq rows are zero) and each key tile starts at a later Q
    tile; with Nq < Nk every query sees the first Nk - Nq keys."""
    for Nq, Nk in ((384, 128), (128, 384)):
        q, k, v = W.make_qkv(1, 2, Nq, Nk, 64, seed=Nq + Nk)
        do = make_dout(1, 2, Nq, 64, seed=7)
        got = gpu_grads(fa, q, k, v, do, 0.125, True)
        ref = AG.attention_grad(q, k, v, do, 0.125, True)
        compare_grads(got, ref, f"Nq={Nq} Nk={Nk} causal")


def test_backward_scale_zero(fa):
    """Uniform weights: dq = dk = 0 exactly, dv spreads dO evenly (oracle closed form)."""
    q, k, v = W.make_qkv(1, 1, 200, 150, 64, seed=9)
    do = make_dout(1, 1, 200, 64, seed=10)
    got = gpu_grads(fa, q, k, v, do, 0.0, True)
    assert np.abs(got[0]).max() == 0 and np.abs(got[1]).max() == 0
    ref = AG.attention_grad(q, k, v, do, 0.0, True)
    compare_grads(got, ref, "scale 0")


def test_backward_deterministic_dk_dv(fa):
    """dK and dV accumulate in one CTA in a fixed order: bit-identical across runs
    (dQ is summed with atomics across key tiles and may differ in the last bits)."""
    q, k, v = W.make_qkv(2, 4, 640, 640, 128, seed=11)
    do = make_dout(2, 4, 640, 128, seed=12)
    dq_, dk_, dv_, do_ = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.fwd(dq_, dk_, dv_, causal=True)
    a = fa.bwd(dq_, dk_, dv_, o, lse, do_, causal=True)
    b = fa.bwd(dq_, dk_, dv_, o, lse, do_, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert (a[0].float() - b[0].float()).abs().max().item() <= 2e-2 * a[0].float().abs().max().item()


def test_backward_rejects(fa):
    x = torch.zeros(1, 1, 8, 96, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 8, dtype=torch.float32, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.bwd(x, x, x, x, lse, x)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    y = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.bwd(y, y, y, y, lse, y, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == fa.FA_ERR_WORKSPACE


@pytest.mark.parametrize("name", ["prefill_2k", "prefill_8k"])
def test_backward_full_size(fa, name):
    """The workloads the benchmark's backward leg times, with its inputs (q, k, v
    seed 0, dO seed 2000): every gradient of two whole heads per causal mode
    (first and last (b, h)) against the fp64 oracle."""
    w = W.WORKLOADS[name]
    q, k, v = W.make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, seed=0)
    gen = torch.Generator().manual_seed(2000)
    do = torch.randn(tuple(q.shape), generator=gen).to(torch.bfloat16)
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    for causal in w.causal_modes:
        o, lse = fa.fwd(qc, kc, vc, scale=w.scale, causal=causal)
        gq, gk, gv = fa.bwd(qc, kc, vc, o, lse, dc, scale=w.scale, causal=causal)
        torch.cuda.synchronize()
        assert fa.device_status() == fa.FA_OK
        for b, h in ((0, 0), (w.B - 1, w.H - 1)):
            got = [t[b, h].double().cpu().numpy() for t in (gq, gk, gv)]
            ref = AG.attend_head_grad(q[b, h], k[b, h], v[b, h], do[b, h], w.scale, causal)
            print(name, causal, (b, h), compare_grads(got, ref, f"{name} causal={causal} head {(b, h)}"))
