"""Host-side checks of the seeded input generator (CPU only)."""

import numpy as np
import torch

from io_aware_exact_fa_gb300 import workloads as W


def test_seeded_and_ordered():
    a = W.make_qkv(1, 2, 5, 7, 8, seed=0)
    b = W.make_qkv(1, 2, 5, 7, 8, seed=0)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and torch.equal(x, y)
    # drawn in the order q, k, v from one generator, then rounded to bf16
    g = torch.Generator().manual_seed(0)
    q = torch.randn(1, 2, 5, 8, generator=g)
    k = torch.randn(1, 2, 7, 8, generator=g)
    assert torch.equal(a[0], q.to(torch.bfloat16)) and torch.equal(a[1], k.to(torch.bfloat16))
    c = W.make_qkv(1, 2, 5, 7, 8, seed=1)
    assert not torch.equal(a[0], c[0])


def test_pack_unpack_roundtrip():
    g = torch.Generator().manual_seed(3)
    for Nk in (1, 31, 32, 33, 100, 128):
        keep = torch.rand(2, 3, 4, Nk, generator=g) < 0.5
        words = W.pack_keep_bits(keep)
        assert words.dtype == torch.int32 and words.shape == (2, 3, 4, (Nk + 31) // 32)
        assert torch.equal(W.unpack_keep_bits(words, Nk), keep)
        # bit (j % 32) of word (j // 32) is key j
        j = Nk - 1
        w = int(words[0, 0, 0, j // 32]) & 0xFFFFFFFF
        assert ((w >> (j % 32)) & 1) == int(keep[0, 0, 0, j])
    full = W.pack_keep_bits(torch.ones(1, 40, dtype=torch.bool))
    assert int(full[0, 0]) == -1 and int(full[0, 1]) == 0xFF


def test_pr1_offsets_are_row_constants():
    q, k, v = W.make_qkv(1, 1, 128, 128, 64)
    q2, k2 = W.add_row_offsets(q, k, 1.0 / 8.0)
    assert torch.all(k2[..., -1] == 1.0)
    s0 = (q.double() @ k2.double().transpose(-1, -2)) / 8.0
    s1 = (q2.double() @ k2.double().transpose(-1, -2)) / 8.0
    diff = (s1 - s0)[0, 0]
    for r, sgn in zip(W.PR1_OFFSET_ROWS, W.PR1_OFFSET_SIGNS):
        row = diff[r]
        assert torch.all(row == row[0])                 # one constant per row
        assert abs(float(row[0]) - sgn * 1e3) < 5.0     # about +/-1e3 after bf16 rounding
    others = [i for i in range(128) if i not in W.PR1_OFFSET_ROWS]
    assert torch.all(diff[others] == 0)


def test_masks_and_strides():
    keep = W.pr1_keep()
    assert keep.shape == (1, 1, 128, 128) and not keep[0, 0, 64].any() and keep[0, 0, 63].all()
    words = W.pack_keep_bits(keep)
    assert W.mask_strides(words) == (128 * 4, 128 * 4, 4)
    kp = W.key_padding_keep(1, 8, 32768, 4, 24576)
    assert kp.shape == (1, 8, 1, 32768)
    assert not kp[0, 3, 0, 24576:].any() and kp[0, 3, 0, :24576].all() and kp[0, 4].all()
    assert W.mask_strides(W.pack_keep_bits(kp))[2] == 0


def test_workload_accounting():
    w = W.WORKLOADS["prefill_2k"]
    assert w.flops(False) == 4 * 4 * 16 * 2048 * 2048 * 64
    assert w.flops(True) == w.flops(False) / 2
    d = W.WORKLOADS["decode_8k"]
    assert d.Nq == 1 and d.num_splits == 16
    kv = 2 * 64 * 32 * 8192 * 128 * 2
    assert kv == 8589934592
    assert d.io_bytes() == kv + 2 * 64 * 32 * 128 * 2 + 4 * 64 * 32


def test_sample_rows():
    r = W.sample_rows(1000, 50, seed=1)
    assert r.shape == (50,) and len(set(r.tolist())) == 50 and torch.all(r[1:] > r[:-1])
    assert torch.equal(r, W.sample_rows(1000, 50, seed=1))


def test_backward_flop_convention():
    w = W.WORKLOADS["prefill_8k"]
    # five products of 2*Nq*Nk*d per (b, h): 2.5x the forward's two
    assert w.bwd_flops(False) == 10 * 1 * 32 * 8192 * 8192 * 128
    assert w.bwd_flops(True) == w.bwd_flops(False) / 2


def test_decode_variant_inputs():
    import dataclasses
    w = dataclasses.replace(W.DECODE_VARIANTS["gqa_spec"], B=3, Nk=512, len_lo=200)
    q, k, v, lens = W.make_decode_inputs(w, seed=5)
    assert q.shape == (3, 32, 4, 128) and k.shape == (3, 8, 512, 128) and v.shape == k.shape
    assert q.dtype == torch.bfloat16 and lens.dtype == torch.int32 and lens.shape == (3,)
    assert int(lens.min()) >= 200 and int(lens.max()) <= 512
    again = W.make_decode_inputs(w, seed=5)
    assert all(torch.equal(a, b) for a, b in zip((q, k, v, lens), again))
    # q, k, v come first from the generator, exactly as make_qkv draws them for a square case
    g = torch.Generator().manual_seed(5)
    assert torch.equal(q, torch.randn(3, 32, 4, 128, generator=g).to(torch.bfloat16))


def test_decode_variant_bytes():
    w = W.DECODE_VARIANTS["gqa"]
    lens = [4096, 8192, 0, 9000]  # clamped to [0, Nk]
    kv = 2 * w.Hkv * w.d * 2 * (4096 + 8192 + 0 + 8192)
    assert w.io_bytes(lens) == kv + 2 * w.B * w.H * w.Nq * w.d * 2 + 4 * w.B * w.H * w.Nq
