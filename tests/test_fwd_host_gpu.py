"""GPU parity of the host-buffer forward pass (fa_fwd_host).

The inputs and outputs live in host memory. The library streams chunks of
heads through two device buffer sets and runs the fused kernel on each chunk.
The results must match the fp64 oracle within the forward tolerances. They
must also be bit-identical to fa_fwd on device copies of the same inputs: each
head's arithmetic does not depend on which other heads share its launch.
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


def _oracle(q, k, v, scale, causal):
    ref = oracle_heads(q, k, v, scale, causal)
    B, H = q.shape[:2]
    ro = np.stack([np.stack([ref[(b, h)][0] for h in range(H)]) for b in range(B)])
    rl = np.stack([np.stack([ref[(b, h)][1] for h in range(H)]) for b in range(B)])
    return ro, rl


# B, H, Nq, Nk, chunk_heads (0 = default): chunks that divide B*H, that leave
# a short last chunk, one head per chunk, and one chunk for everything
CASES = [(2, 3, 300, 300, 0), (1, 5, 200, 457, 2), (3, 2, 129, 129, 1), (2, 2, 260, 140, 100)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}q{}k{}c{}".format(*c))
def test_fwd_host_vs_oracle(fa, case, d):
    B, H, Nq, Nk, ch = case
    q, k, v = W.make_qkv(B, H, Nq, Nk, d, seed=B * 100 + H + d)
    scale = 1.0 / math.sqrt(d)
    qp, kp, vp = q.pin_memory(), k.pin_memory(), v.pin_memory()
    for causal in (False, True):
        o, lse = fa.fwd_host(qp, kp, vp, scale=scale, causal=causal, chunk_heads=ch)
        assert fa.device_status() == fa.FA_OK
        assert o.device.type == "cpu" and o.is_pinned()
        ro, rl = _oracle(q, k, v, scale, causal)
        print(case, d, causal, compare(to64(o), to64(lse), ro, rl, f"{case} d={d} causal={causal}"))
        od, ld = fa.fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())


def test_fwd_host_pageable_and_no_lse(fa):
    """Pageable host memory gives the same bytes; lse may be left out."""
    q, k, v = W.make_qkv(1, 4, 333, 333, 64, seed=9)
    o1, l1 = fa.fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), causal=True, chunk_heads=3)
    o2, l2 = fa.fwd_host(q, k, v, causal=True, chunk_heads=3)
    o3, l3 = fa.fwd_host(q, k, v, causal=True, chunk_heads=3, with_lse=False)
    assert l3 is None
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(o1, o3)


def test_fwd_host_stream_ordering(fa):
    """Several calls queued on one non-default stream without synchronising,
    sharing one workspace: each call's chunks wait for the previous call's, so
    every output is that of its own inputs."""
    s = torch.cuda.Stream()
    ins = [W.make_qkv(2, 4, 256, 384, 128, seed=40 + i) for i in range(3)]
    ws = torch.empty(fa.fwd_host_workspace_size(2, 4, 256, 384, 128, 3), dtype=torch.uint8, device="cuda")
    outs = []
    for q, k, v in ins:
        outs.append(fa.fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), causal=True, chunk_heads=3,
                                workspace=ws, stream=s, sync=False))
    s.synchronize()
    assert fa.device_status() == fa.FA_OK
    for (q, k, v), (o, lse) in zip(ins, outs):
        od, ld = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
        torch.cuda.synchronize()
        assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_host_2k_d64_full_size(fa, causal):
    """The benchmark workload (B=4 H=16 N=2048 d=64, seed 0) with the default
    chunking: bit-identical to fa_fwd, and two whole heads against the oracle."""
    w = W.WORKLOADS["prefill_2k"]
    q, k, v = W.make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, seed=0)
    o, lse = fa.fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), scale=w.scale, causal=causal)
    assert fa.device_status() == fa.FA_OK
    od, ld = fa.fwd(q.cuda(), k.cuda(), v.cuda(), scale=w.scale, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    ref = oracle_heads(q, k, v, w.scale, causal, heads=heads)
    for b, h in heads:
        compare(to64(o[b, h]), to64(lse[b, h]), ref[(b, h)][0], ref[(b, h)][1], f"head {b},{h} causal={causal}")


def test_fwd_host_rejects(fa):
    q = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):  # device tensors are not host buffers
        fa.fwd_host(q.cuda(), q.cuda(), q.cuda())
    with pytest.raises(fa.FAError) as e:
        fa.fwd_host(q, q, q, workspace=torch.empty(64, dtype=torch.uint8, device="cuda"))
    assert e.value.status == fa.FA_ERR_WORKSPACE
