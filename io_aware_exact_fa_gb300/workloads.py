"""Seeded synthetic inputs for the attention forward pass and split-KV decode.

This module only draws random numbers and packs masks; it holds none of the
attention arithmetic. Tests and the benchmark feed the SAME bytes it produces
to the CUDA path and to the fp64 oracle.

Recipe: ``torch.randn`` in fp32 from a generator seeded with ``seed``, drawn in
the order q, k, v, then rounded to bf16 (round-to-nearest-even). Large
workloads can be drawn directly on a CUDA device (same recipe, the device's
Philox generator); the oracle then receives sampled slices copied back.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    scale: float
    causal_modes: Tuple[bool, ...] = (False,)
    kind: str = "prefill"           # "prefill" or "decode"
    num_splits: int = 0             # decode only
    pad_heads: int = 0              # heads h < pad_heads get key padding ...
    pad_from: int = 0               # ... masking keys j >= pad_from

    def flops(self, causal: bool) -> float:
        """Algorithmic FLOPs of the two products: 4*B*H*Nq*Nk*d, halved for causal."""
        f = 4.0 * self.B * self.H * self.Nq * self.Nk * self.d
        return f / 2 if causal else f

    def bwd_flops(self, causal: bool) -> float:
        """Algorithmic FLOPs of the backward pass's five products (S recomputed,
        dP, dV, dK, dQ, each 2*Nq*Nk*d per head): 2.5x the forward's, halved for causal."""
        return 2.5 * self.flops(causal)

    def io_bytes(self) -> int:
        """Minimum HBM bytes: Q, K, V read once and O written once (2-byte
        elements) plus the fp32 per-row log-sum-exp."""
        qo = 2 * self.B * self.H * self.Nq * self.d * 2
        kv = 2 * self.B * self.H * self.Nk * self.d * 2
        return qo + kv + 4 * self.B * self.H * self.Nq


WORKLOADS = {
    # 1 head, 128 x 128, d = 64; rows 124..127 carry a +/-1e3 additive score
    # offset (see ``offset_rows``), row 64 is fully key-masked.
    "pr1": Workload("pr1_b1h1n128d64", 1, 1, 128, 128, 64, 1.0 / 8.0, (False, True)),
    "prefill_2k": Workload("prefill_b4h16n2048d64", 4, 16, 2048, 2048, 64, 1.0 / 8.0, (False, True)),
    "prefill_8k": Workload("prefill_b1h32n8192d128_causal", 1, 32, 8192, 8192, 128,
                           1.0 / math.sqrt(128.0), (True,)),
    "prefill_32k": Workload("prefill_b1h8n32768d128_causal", 1, 8, 32768, 32768, 128,
                            1.0 / math.sqrt(128.0), (True,)),
    "prefill_32k_pad": Workload("prefill_b1h8n32768d128_causal_keypad", 1, 8, 32768, 32768, 128,
                                1.0 / math.sqrt(128.0), (True,), pad_heads=4, pad_from=24576),
    "decode_8k": Workload("decode_b64h32nk8192d128_split16", 64, 32, 1, 8192, 128,
                          1.0 / math.sqrt(128.0), (False,), kind="decode", num_splits=16),
}

@dataclasses.dataclass(frozen=True)
class DecodeVariant:
    """Decode with grouped K/V heads, Nq new tokens per sequence and ragged
    per-sequence KV lengths drawn uniformly from [len_lo, Nk] (seeded)."""
    name: str
    B: int
    H: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    scale: float
    num_splits: int
    len_lo: int

    def io_bytes(self, seqlens: Sequence[int]) -> int:
        """Minimum HBM bytes: the visible K and V rows of every sequence read
        once, q and o (2-byte elements) and the fp32 lse."""
        kv = 2 * self.Hkv * self.d * 2 * int(sum(min(max(int(x), 0), self.Nk) for x in seqlens))
        qo = 2 * self.B * self.H * self.Nq * self.d * 2
        return kv + qo + 4 * self.B * self.H * self.Nq


DECODE_VARIANTS = {
    # 4 query heads per K/V head, one new token, ragged lengths in [4096, 8192]
    "gqa": DecodeVariant("decode_gqa_b64h32kv8nq1_nk8192d128_ragged", 64, 32, 8, 1, 8192, 128,
                         1.0 / math.sqrt(128.0), 4, 4096),
    # the same with 4 new (speculative) tokens per sequence
    "gqa_spec": DecodeVariant("decode_gqa_b64h32kv8nq4_nk8192d128_ragged", 64, 32, 8, 4, 8192, 128,
                              1.0 / math.sqrt(128.0), 4, 4096),
    # one and four new tokens at head dim 64 (the prefill workload's head dim)
    "gqa_d64": DecodeVariant("decode_gqa_b64h32kv8nq1_nk8192d64_ragged", 64, 32, 8, 1, 8192, 64,
                             1.0 / 8.0, 4, 4096),
    "gqa_spec_d64": DecodeVariant("decode_gqa_b64h32kv8nq4_nk8192d64_ragged", 64, 32, 8, 4, 8192, 64,
                                  1.0 / 8.0, 4, 4096),
}


def make_decode_inputs(w: DecodeVariant, seed: int = 0, device: str = "cpu"):
    """q [B,H,Nq,d], k/v [B,Hkv,Nk,d] bf16 (order q, k, v) and seqlens int32 [B]
    uniform in [len_lo, Nk], drawn after v from the same generator."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    q = torch.randn(w.B, w.H, w.Nq, w.d, generator=g, device=device, dtype=torch.float32)
    k = torch.randn(w.B, w.Hkv, w.Nk, w.d, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(w.B, w.Hkv, w.Nk, w.d, generator=g, device=device, dtype=torch.float32)
    lens = torch.randint(w.len_lo, w.Nk + 1, (w.B,), generator=g, device=device, dtype=torch.int32)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16), lens


PR1_OFFSET_ROWS = (124, 125, 126, 127)
PR1_OFFSET_SIGNS = (+1.0, -1.0, +1.0, -1.0)
PR1_OFFSET = 1.0e3
PR1_MASKED_ROW = 64


def make_qkv(B: int, H: int, Nq: int, Nk: int, d: int, seed: int = 0,
             device: str = "cpu") -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """q [B,H,Nq,d], k/v [B,H,Nk,d], bf16, N(0,1) before rounding; order q, k, v."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    q = torch.randn(B, H, Nq, d, generator=g, device=device, dtype=torch.float32)
    k = torch.randn(B, H, Nk, d, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(B, H, Nk, d, generator=g, device=device, dtype=torch.float32)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


E4M3_MAX = 448.0  # largest finite e4m3 magnitude


def make_qkv_fp8(B: int, H: int, Nq: int, Nk: int, d: int, seed: int = 0, device: str = "cpu"):
    """FP8 inputs: the fp32 N(0,1) draws of ``make_qkv`` (same seed, same
    order q, k, v), each tensor quantized to e4m3 with one descale factor
    amax / 448 (so its largest magnitude maps to the largest e4m3 value,
    round-to-nearest-even by torch's float8_e4m3fn conversion). Returns
    (q8, k8, v8) as uint8 code tensors and (descale_q, descale_k, descale_v)
    as Python floats."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out, ds = [], []
    for n in (Nq, Nk, Nk):
        x = torch.randn(B, H, n, d, generator=g, device=device, dtype=torch.float32)
        amax = float(x.abs().max()) if x.numel() else 1.0
        descale = amax / E4M3_MAX if amax > 0 else 1.0
        out.append((x / descale).to(torch.float8_e4m3fn).view(torch.uint8).contiguous())
        ds.append(descale)
    return tuple(out), tuple(ds)


def add_row_offsets(q: torch.Tensor, k: torch.Tensor, scale: float,
                    rows: Sequence[int] = PR1_OFFSET_ROWS,
                    signs: Sequence[float] = PR1_OFFSET_SIGNS,
                    offset: float = PR1_OFFSET) -> Tuple[torch.Tensor, torch.Tensor]:
    """Give ``rows`` an additive score offset of about +/-``offset`` through Q.

    The last key component is set to exactly 1 for every key and
    ``sign*offset/scale`` is added to the last component of each chosen query
    row, so every score of that row moves by the same constant (the bf16
    rounding of the shifted query entry makes the constant inexact, but it is
    still one constant per row). Returns new bf16 tensors.
    """
    q = q.clone()
    k = k.clone()
    k[..., -1] = 1.0
    qf = q.float()
    for r, sgn in zip(rows, signs):
        qf[..., r, -1] += sgn * offset / scale
    return qf.to(torch.bfloat16), k


def scale_rows(q: torch.Tensor, factors: Sequence[float], rows: Sequence[int]) -> torch.Tensor:
    """Multiply chosen query rows by constants (a large score spread), rounded to bf16."""
    qf = q.float().clone()
    for r, f in zip(rows, factors):
        qf[..., r, :] *= f
    return qf.to(torch.bfloat16)


def pack_keep_bits(keep: torch.Tensor) -> torch.Tensor:
    """Pack a bool mask [..., Nk] (True = attend) into int32 words [..., ceil(Nk/32)].

    Bit (j % 32) of word (j // 32) is key j; bits past Nk are zero.
    """
    keep = keep.to(torch.bool)
    Nk = keep.shape[-1]
    W = (Nk + 31) // 32
    pad = W * 32 - Nk
    if pad:
        keep = torch.cat([keep, torch.zeros(*keep.shape[:-1], pad, dtype=torch.bool,
                                            device=keep.device)], dim=-1)
    bits = keep.reshape(*keep.shape[:-1], W, 32).to(torch.int64)
    weights = (torch.ones(32, dtype=torch.int64, device=keep.device) << torch.arange(32, device=keep.device))
    words = (bits * weights).sum(-1)
    # reinterpret the unsigned 32-bit pattern as int32
    words = torch.where(words >= 2**31, words - 2**32, words)
    return words.to(torch.int32).contiguous()


def unpack_keep_bits(words: torch.Tensor, Nk: int) -> torch.Tensor:
    """Inverse of ``pack_keep_bits``: int32 words [..., W] -> bool [..., Nk]."""
    w = words.to(torch.int64) & 0xFFFFFFFF
    bits = (w.unsqueeze(-1) >> torch.arange(32, device=words.device)) & 1
    return bits.reshape(*words.shape[:-1], -1)[..., :Nk].to(torch.bool)


def pr1_keep(Nq: int = 128, Nk: int = 128, masked_row: int = PR1_MASKED_ROW) -> torch.Tensor:
    """Per-row mask [1, 1, Nq, Nk]: every key kept except for one fully masked row."""
    keep = torch.ones(1, 1, Nq, Nk, dtype=torch.bool)
    keep[..., masked_row, :] = False
    return keep


def key_padding_keep(B: int, H: int, Nk: int, pad_heads: int, pad_from: int) -> torch.Tensor:
    """Key-padding mask [B, H, 1, Nk]: heads h < pad_heads drop keys j >= pad_from."""
    keep = torch.ones(B, H, 1, Nk, dtype=torch.bool)
    keep[:, :pad_heads, :, pad_from:] = False
    return keep


def mask_strides(words: torch.Tensor) -> Tuple[int, int, int]:
    """(stride_b, stride_h, stride_q) in words for a packed mask [B, H, Q, W];
    a query extent of 1 broadcasts over rows (stride 0)."""
    B, H, Q, W = words.shape
    sq = 0 if Q == 1 else W
    return (H * Q * W, Q * W, sq)


def sample_rows(Nq: int, count: int, seed: int = 1) -> torch.Tensor:
    """Seeded random subset of query rows (sorted, unique) for sampled parity."""
    g = torch.Generator().manual_seed(seed)
    count = min(count, Nq)
    return torch.randperm(Nq, generator=g)[:count].sort().values
