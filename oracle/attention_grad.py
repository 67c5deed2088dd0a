"""fp64 CPU oracle for the attention backward pass -- TEST INFRASTRUCTURE ONLY.

Only tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may import
this module. It imports nothing from the CUDA path.

What it computes: the gradients of a scalar loss L through O = softmax(S) V,
S = scale * Q K^T + mask, for the cotangent dO = dL/dO, i.e. dL/dQ, dL/dK and
dL/dV. The pages state the training side of the method only in words: the
backward pass needs the probability matrix P again and recomputes its tiles
from the saved per-row statistics instead of storing P ("Flash Attention
Optimization", section "Sizing a tile, and why the backward pass recomputes
instead of storing"; "Explain FlashAttention. Why is it called IO-aware, and
what does it actually save?", section "Exact attention, finite precision and
backward"). The gradients themselves have a plain definition, the chain rule
through the definition of O, and that definition is written out here, with
the exact P of the forward definition:

    dV = P^T dO
    dP = dO V^T
    dS = P * (dP - D),   D_i = sum_j P_ij dP_ij   (softmax Jacobian, row i)
    dQ = scale * dS K
    dK = scale * dS^T Q

Masked (query, key) pairs have P = 0 and so dS = 0; a row with no allowed key
has O = 0 for every input and contributes nothing.
"""

from __future__ import annotations

from typing import Optional, Tuple

import numpy as np

from oracle.attention import _f64, allowed_mask


def attend_head_grad(q, k, v, do, scale: float, causal: bool = False, keep=None,
                     row_block: int = 256) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Gradients for one (batch, head): q [Nq,d], k [Nk,d], v [Nk,dv], do [Nq,dv].

    Returns (dq [Nq,d], dk [Nk,d], dv [Nk,dv]) in fp64. ``keep`` is None or
    bool broadcastable to [Nq, Nk] (True = attend); causal alignment is
    bottom-right (key j visible to query i iff j <= i + Nk - Nq). Query rows
    are processed ``row_block`` at a time only to bound memory.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    Nq, Nk = q.shape[0], k.shape[0]
    if k.shape[1] != q.shape[1] or v.shape[0] != Nk or do.shape != (Nq, v.shape[1]):
        raise ValueError("q/k/v/do shapes disagree")
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    keep_full = None if keep is None else np.broadcast_to(np.asarray(keep, dtype=bool), (Nq, Nk))
    if Nk == 0 or Nq == 0:
        return dq, dk, dv
    for r0 in range(0, Nq, row_block):
        rb = np.arange(r0, min(Nq, r0 + row_block))
        s = scale * (q[rb] @ k.T)
        ok = allowed_mask(rb, Nk, Nq, causal, None if keep_full is None else keep_full[rb])
        s = np.where(ok, s, -np.inf)
        any_ok = ok.any(axis=1)
        M = np.where(any_ok, s.max(axis=1), 0.0)
        w = np.where(ok, np.exp(s - M[:, None]), 0.0)
        L = np.where(any_ok, w.sum(axis=1), 1.0)
        P = w / L[:, None]                       # exact probabilities, 0 where masked
        dv += P.T @ do[rb]
        dP = do[rb] @ v.T
        D = (P * dP).sum(axis=1)
        dS = P * (dP - D[:, None])
        dq[rb] = scale * (dS @ k)
        dk += scale * (dS.T @ q[rb])
    return dq, dk, dv


def attention_grad(q, k, v, do, scale: float, causal: bool = False, keep=None,
                   row_block: int = 256) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Batched: q [B,H,Nq,d], k/v [B,H,Nk,d], do [B,H,Nq,dv] -> (dq, dk, dv), fp64."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, Nq, _ = q.shape
    Nk = k.shape[2]
    kb = None if keep is None else np.broadcast_to(np.asarray(keep, dtype=bool), (B, H, Nq, Nk))
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = attend_head_grad(
                q[b, h], k[b, h], v[b, h], do[b, h], scale, causal,
                None if kb is None else kb[b, h], row_block=row_block)
    return dq, dk, dv
