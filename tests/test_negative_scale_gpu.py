"""GPU parity at a negative softmax scale, against the fp64 oracle.

softmax(scale * Q K^T + mask) V is defined for any finite scale; with scale
< 0 the largest weights go to the smallest dot products. The kernels that
take a row maximum on the tensor cores (prefill, the tensor-core grouped
decode kernels) run such a call as |scale| times scores that the score MMA
negates; the split-KV decode and the CUDA-core grouped decode (d = 64, at
most four query rows per K/V head) scale q itself, and the backward pass
takes no maximum. Every entry point is
checked here on ragged sizes, with the tolerances of the positive-scale
tests.
"""

import math

import numpy as np
import pytest
import torch

from io_aware_exact_fa_gb300 import workloads as W
from oracle import attention as A
from oracle import attention_grad as AG
from oracle import decode_variants as DV
from tests.parity import compare, oracle_heads, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_fa_gb300 import build
    build.build()
    from io_aware_exact_fa_gb300 import fa as lib
    return lib


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_prefill_negative_scale(fa, d, causal):
    B, H, Nq, Nk = 1, 3, 300, 450
    q, k, v = W.make_qkv(B, H, Nq, Nk, d, seed=21)
    keep = torch.ones(B, H, Nq, Nk, dtype=torch.bool)
    keep[0, 1, 7] = False                   # one fully masked row: O = 0, lse = -inf
    keep[0, 2, :, 100:140] = False          # a band of masked keys
    scale = -1.0 / math.sqrt(d)
    words = W.pack_keep_bits(keep)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal, keep_bits=words.cuda(),
                    mask_strides=W.mask_strides(words))
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    ref = oracle_heads(q, k, v, scale, causal, keep)
    ro = np.stack([ref[(0, h)][0] for h in range(H)])[None]
    rl = np.stack([ref[(0, h)][1] for h in range(H)])[None]
    print(compare(to64(o), to64(lse), ro, rl, f"negative scale d={d} causal={causal}"))
    # the sign matters: the same call at +|scale| must give a different result
    o_pos, _ = fa.fwd(q.cuda(), k.cuda(), v.cuda(), scale=-scale, causal=causal)
    torch.cuda.synchronize()
    assert np.abs(to64(o_pos)[0, 0] - ro[0, 0]).max() > 0.05


def test_split_decode_negative_scale(fa):
    B, H, Nk, d, S = 2, 3, 1000, 128, 7
    q, k, v = W.make_qkv(B, H, 1, Nk, d, seed=22)
    scale = -0.09
    o, lse = fa.decode(q.cuda(), k.cuda(), v.cuda(), scale=scale, num_splits=S)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    ro = np.zeros((B, H, 1, d))
    rl = np.zeros((B, H, 1))
    for b in range(B):
        for h in range(H):
            ro[b, h], rl[b, h] = A.attend_head(to64(q[b, h]), to64(k[b, h]), to64(v[b, h]), scale)
    print(compare(to64(o).reshape(B * H, d), to64(lse).reshape(-1), ro.reshape(B * H, d), rl.reshape(-1),
                  "split decode, negative scale"))


@pytest.mark.parametrize("Nq,d", [(3, 128), (1, 128), (1, 64)])
def test_grouped_decode_negative_scale(fa, Nq, d):
    g = torch.Generator().manual_seed(23)
    B, H, Hkv, Nk = 2, 8, 2, 300
    q = torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, Nk, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, Nk, d, generator=g).to(torch.bfloat16)
    lens = [300, 57]
    scale = -1.0 / math.sqrt(d)
    o, lse = fa.decode_grouped(q.cuda(), k.cuda(), v.cuda(),
                               seqlens_k=torch.tensor(lens, dtype=torch.int32).cuda(), scale=scale, num_splits=2)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    ro, rl = DV.decode_grouped_attention(q, k, v, lens, scale)
    print(compare(to64(o).reshape(-1, d), to64(lse).reshape(-1), ro.reshape(-1, d), rl.reshape(-1),
                  "grouped decode, negative scale"))


@pytest.mark.parametrize("causal", [False, True])
def test_backward_negative_scale(fa, causal):
    B, H, Nq, Nk, d = 1, 2, 200, 260, 64
    q, k, v = W.make_qkv(B, H, Nq, Nk, d, seed=24)
    do = torch.randn(B, H, Nq, d, generator=torch.Generator().manual_seed(25)).to(torch.bfloat16)
    scale = -0.125
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.fwd(qc, kc, vc, scale=scale, causal=causal)
    grads = fa.bwd(qc, kc, vc, o, lse, do.cuda(), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    refs = AG.attention_grad(q, k, v, do, scale, causal)
    for name, gpu, ref in zip(("dq", "dk", "dv"), grads, refs):
        diff = np.abs(to64(gpu) - ref)
        assert diff.max() <= 2e-2 * np.abs(ref).max(), name
        assert diff.mean() <= 1e-2 * np.abs(ref).mean(), name
