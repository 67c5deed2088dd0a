"""GPU parity of split-KV decode (split kernel + merge kernel) against the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

from io_aware_exact_fa_gb300 import workloads as W
from oracle import attention as A
from tests.parity import compare, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_fa_gb300 import build
    build.build()
    from io_aware_exact_fa_gb300 import fa as lib
    return lib


def run(fa, q, k, v, scale, splits):
    o, lse = fa.decode(q.cuda(), k.cuda(), v.cuda(), scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    return to64(o), to64(lse)


def oracle(q, k, v, scale, heads=None):
    B, H = q.shape[:2]
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    o = np.stack([A.attend_head(to64(q[b, h]), to64(k[b, h]), to64(v[b, h]), scale)[0][0] for b, h in heads])
    l = np.stack([A.attend_head(to64(q[b, h]), to64(k[b, h]), to64(v[b, h]), scale)[1][0] for b, h in heads])
    return o, l


CASES = [(1, 1, 1, 1), (1, 1, 5, 16), (2, 3, 100, 7), (2, 2, 513, 16), (1, 4, 1000, 3), (3, 2, 4096, 16),
         (1, 1, 64, 64), (2, 1, 8192, 1)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_decode_small(fa, case, d):
    B, H, Nk, S = case
    q, k, v = W.make_qkv(B, H, 1, Nk, d, seed=Nk + S)
    scale = 1 / math.sqrt(d)
    o, lse = run(fa, q, k, v, scale, S)
    ro, rl = oracle(q, k, v, scale)
    compare(o.reshape(B * H, d), lse.reshape(-1), ro, rl, f"decode {case} d={d}")


def test_decode_splits_agree_with_merge_oracle(fa):
    """The GPU result for any number of splits equals the oracle's own split+merge."""
    q, k, v = W.make_qkv(2, 2, 1, 777, 128, seed=3)
    ro, rl = A.splitkv_attention(to64(q), to64(k), to64(v), 0.09, 5)
    for S in (1, 2, 5, 16, 64, 777, 1024):
        o, lse = run(fa, q, k, v, 0.09, S)
        compare(o.reshape(4, 128), lse.reshape(-1), ro.reshape(4, 128), rl.reshape(-1), f"S={S}")


def test_decode_offsets(fa):
    """Large additive score offsets (via a constant key column) do not change O."""
    q, k, v = W.make_qkv(1, 4, 1, 2048, 128, seed=4)
    k = k.clone()
    k[..., -1] = 1.0
    o0, l0 = run(fa, q, k, v, 1 / math.sqrt(128), 16)
    q2 = q.float().clone()
    q2[:, :, 0, -1] += torch.tensor([1e3, -1e3, 5e2, -5e2]) * math.sqrt(128)
    o1, l1 = run(fa, q2.to(torch.bfloat16), k, v, 1 / math.sqrt(128), 16)
    assert np.abs(o1 - o0).max() < 1e-2


def test_decode_full_size_sampled(fa):
    """B=64, H=32, Nk=8192, d=128, 16 splits; inputs drawn on the device,
    64 seeded (b, h) heads compared against the oracle."""
    w = W.WORKLOADS["decode_8k"]
    q, k, v = W.make_qkv(w.B, w.H, 1, w.Nk, w.d, seed=0, device="cuda")
    o, lse = fa.decode(q, k, v, scale=w.scale, num_splits=w.num_splits)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    g = torch.Generator().manual_seed(2)
    idx = torch.randperm(w.B * w.H, generator=g)[:64].tolist()
    heads = sorted({(i // w.H, i % w.H) for i in idx} | {(0, 0), (w.B - 1, w.H - 1)})
    qs = torch.stack([q[b, h] for b, h in heads]).cpu()
    ks = torch.stack([k[b, h] for b, h in heads]).cpu()
    vs = torch.stack([v[b, h] for b, h in heads]).cpu()
    ro = np.stack([A.attend_head(to64(qs[i]), to64(ks[i]), to64(vs[i]), w.scale)[0][0] for i in range(len(heads))])
    rl = np.stack([A.attend_head(to64(qs[i]), to64(ks[i]), to64(vs[i]), w.scale)[1][0] for i in range(len(heads))])
    go = np.stack([to64(o[b, h, 0]) for b, h in heads])
    gl = np.stack([float(lse[b, h]) for b, h in heads])
    print(compare(go, gl, ro, rl, "decode full size"))


def test_decode_workspace_errors(fa):
    q, k, v = W.make_qkv(1, 1, 1, 64, 64, seed=0)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.decode(q.cuda(), k.cuda(), v.cuda(), workspace=small)
    assert e.value.status == fa.FA_ERR_WORKSPACE
