"""fp64 CPU oracle for the decode variants -- TEST INFRASTRUCTURE ONLY.

Only tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may import
this module. It imports nothing from the CUDA path.

What it computes: decode attention for
  * grouped K/V heads: H query heads share Hkv K/V heads, query head h reads
    K/V head h // (H / Hkv);
  * several new query tokens per sequence: the Nq tokens are the last Nq
    positions of the sequence, so token t sees key j iff j <= L_b - Nq + t;
  * per-sequence KV lengths: sequence b holds only its first L_b keys.
Decode is attention of the new tokens over the cache ("FlashAttention:
Attention Is Limited by Memory, Not Math", section "Where it helps, and where
it does not"); the causal rule uses absolute positions ("Explain
FlashAttention ...", the note that the causal mask uses absolute query and
key positions). With keys cut to the first L_b, that rule is the forward
oracle's bottom-right causal alignment (key j visible to query i iff
j <= i + Nk - Nq) with Nk = L_b, so each (b, h) is one call of the pinned
forward definition on the sequence's visible prefix. A token that sees no key
gets O = 0 and lse = -inf.
"""

from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np

from oracle.attention import _f64, attend_head


def decode_grouped_attention(q, k, v, seqlens: Optional[Sequence[int]], scale: float,
                             heads: Optional[Sequence[Tuple[int, int]]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """q [B,H,Nq,d], k/v [B,Hkv,Nk,d], seqlens: B lengths (None: all Nk; clamped to [0, Nk]).

    Returns (O [B,H,Nq,d], lse [B,H,Nq]) in fp64. ``heads``, if given, limits
    the work to those (b, h) pairs; the other entries are left as NaN.
    """
    # numpy or torch inputs; each head is converted to fp64 (exactly) as it is used
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if H % Hkv != 0:
        raise ValueError("H must be a multiple of Hkv")
    G = H // Hkv
    o = np.full((B, H, Nq, v.shape[3]), np.nan)
    lse = np.full((B, H, Nq), np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        L = Nk if seqlens is None else min(max(int(seqlens[b]), 0), Nk)
        g = h // G
        o[b, h], lse[b, h] = attend_head(_f64(q[b, h]), _f64(k[b, g, :L]), _f64(v[b, g, :L]), scale, causal=True)
    return o, lse
