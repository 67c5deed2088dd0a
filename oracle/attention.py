"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this module. It imports nothing from the CUDA path.

Sources (web pages, cited by title and section):

[FAO]  "Flash Attention Optimization" -- sections "Attention is not slow
       because of arithmetic" (S = Q K^T / sqrt(d), P = softmax(S), O = P V),
       "The fix: tile the computation, never materialize the full matrix"
       (block-local-max recurrence), "Worked example: online softmax by hand",
       "Tracing the algorithm as code".
[MEM]  "FlashAttention: Attention Is Limited by Memory, Not Math" -- sections
       "How tiling and online softmax stay exact" (running max and sum, rescale
       by exp(m_old - m_new)), "Where it helps, and where it does not"
       (split-KV decode merges partial results), "Try it" (new-max tiled form).
[NOTES] "Handwritten Notes on Flash Attention" -- section "Merging two blocks"
       (re-basing a block to a new max is one scalar per block; the merge is
       associative and continues over N/B blocks).
[IO]   "Explain FlashAttention. Why is it called IO-aware, and what does it
       actually save?" -- sections "Keep only the state needed for the final
       weighted average" (scores = q K^T / sqrt(d) plus mask or bias; new-max
       recurrence with alpha = exp(m - m_new)), "Executable recurrence, with an
       empty-state policy" (input checks, skip all-masked chunks, all-masked
       row returns zeros), and the causal-mask remark that follows it (the mask
       uses absolute query and key positions).

Readings taken where the pages are silent (each one is also listed with the
design notes of the repository):

* lse is the natural-log log-sum-exp of the scaled, masked scores of a row,
  lse = m + ln(l); an all-masked row has lse = -inf and output 0.
* causal alignment when Nq != Nk is bottom-right: key j is visible to query i
  iff j <= i + (Nk - Nq); for Nq == Nk this is the usual j <= i.
* ``keep`` is a boolean mask broadcastable to [B, H, Nq, Nk]; True = attend.
"""

from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    """Exact conversion of any real array (numpy, or torch via .numpy()) to fp64."""
    if hasattr(x, "detach"):  # a torch tensor; bf16 has no numpy dtype
        import torch

        x = x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# The plain definition
# ---------------------------------------------------------------------------

def allowed_mask(rows: np.ndarray, Nk: int, Nq: int, causal: bool,
                 keep_rows: Optional[np.ndarray]) -> np.ndarray:
    """Boolean [len(rows), Nk]: which keys each query row may attend to.

    Causal masking uses absolute positions [IO, causal remark]; with the
    bottom-right reading key j is visible to query i iff j <= i + (Nk - Nq).
    ``keep_rows`` (already sliced to these rows, broadcastable) ANDs in an
    arbitrary key mask [IO, "Keep only the state ..." -- "plus the intended
    mask or bias"].
    """
    rows = np.asarray(rows)
    allowed = np.ones((rows.shape[0], Nk), dtype=bool)
    if causal:
        j = np.arange(Nk)[None, :]
        allowed &= j <= (rows[:, None] + (Nk - Nq))
    if keep_rows is not None:
        allowed &= np.broadcast_to(np.asarray(keep_rows, dtype=bool), allowed.shape)
    return allowed


def attend_head(q, k, v, scale: float, causal: bool = False, keep=None,
                rows: Optional[Sequence[int]] = None,
                row_block: int = 256) -> Tuple[np.ndarray, np.ndarray]:
    """Exact attention for one (batch, head): O = softmax(scale * q k^T + mask) v.

    q: [Nq, d], k: [Nk, d], v: [Nk, dv]; keep: None or bool broadcastable to
    [Nq, Nk]; rows: optional subset of query indices (default all).
    Returns (O [len(rows), dv], lse [len(rows)]), both fp64.

    This is the definition written out [FAO, "Attention is not slow because of
    arithmetic"; IO, "Keep only the state ..."]: for each row, the scaled
    scores s_j = scale * <q_i, k_j>; over the allowed keys M = max s_j,
    w_j = exp(s_j - M) (the stable softmax), L = sum w_j, O_i = sum w_j v_j / L,
    lse_i = M + ln L. A row with no allowed key returns O = 0, lse = -inf
    [IO, "Executable recurrence, with an empty-state policy"]. Rows are
    processed ``row_block`` at a time only to bound memory; no score matrix
    larger than row_block x Nk is ever formed.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Nq, Nk = q.shape[0], k.shape[0]
    if k.shape[1] != q.shape[1] or v.shape[0] != Nk:
        raise ValueError("q/k head dims or k/v lengths disagree")
    rows = np.arange(Nq) if rows is None else np.asarray(rows, dtype=np.int64)
    dv = v.shape[1]
    out = np.zeros((rows.shape[0], dv))
    lse = np.full(rows.shape[0], NEG_INF)
    keep_full = None
    if keep is not None:
        keep_full = np.broadcast_to(np.asarray(keep, dtype=bool), (Nq, Nk))
    if Nk == 0:
        return out, lse
    for r0 in range(0, rows.shape[0], row_block):
        rb = rows[r0:r0 + row_block]
        s = scale * (q[rb] @ k.T)                       # [rb, Nk] scaled scores
        ok = allowed_mask(rb, Nk, Nq, causal,
                          None if keep_full is None else keep_full[rb])
        s = np.where(ok, s, NEG_INF)
        any_ok = ok.any(axis=1)
        M = np.where(any_ok, s.max(axis=1), 0.0)         # row max over allowed keys
        w = np.where(ok, np.exp(s - M[:, None]), 0.0)    # stable exponentials
        L = w.sum(axis=1)
        num = w @ v
        safe_L = np.where(any_ok, L, 1.0)
        out[r0:r0 + rb.shape[0]] = np.where(any_ok[:, None], num / safe_L[:, None], 0.0)
        lse[r0:r0 + rb.shape[0]] = np.where(any_ok, M + np.log(safe_L), NEG_INF)
    return out, lse


def naive_attention(q, k, v, scale: float, causal: bool = False, keep=None,
                    row_block: int = 256) -> Tuple[np.ndarray, np.ndarray]:
    """Batched plain definition: q [B,H,Nq,d], k/v [B,H,Nk,d] -> (O [B,H,Nq,dv], lse [B,H,Nq]).

    ``keep`` is None or bool broadcastable to [B, H, Nq, Nk] (True = attend).
    Real implementations put batch and head dimensions on top of the
    single-sequence algorithm [NOTES, "Algorithm 1, annotated"]; each (b, h)
    is independent.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, _ = q.shape
    Nk = k.shape[2]
    out = np.zeros((B, H, Nq, v.shape[3]))
    lse = np.full((B, H, Nq), NEG_INF)
    kb = None if keep is None else np.broadcast_to(np.asarray(keep, dtype=bool), (B, H, Nq, Nk))
    for b in range(B):
        for h in range(H):
            out[b, h], lse[b, h] = attend_head(
                q[b, h], k[b, h], v[b, h], scale, causal,
                None if kb is None else kb[b, h], row_block=row_block)
    return out, lse


# ---------------------------------------------------------------------------
# The tile-by-tile online recurrence (new-max form)
# ---------------------------------------------------------------------------

def online_attention_head(q, k, v, scale: float, causal: bool = False, keep=None,
                          tile: int = 128) -> Tuple[np.ndarray, np.ndarray]:
    """One head by the online recurrence over key tiles of size ``tile``.

    State per query row [IO, "Keep only the state ..."; MEM, "Try it"]:
    running max m (init -inf), running sum l (init 0), unnormalised output o
    (init 0). For each key tile with scaled, masked scores s:
        m_new = max(m, max(s)); alpha = exp(m - m_new); p = exp(s - m_new)
        l = alpha * l + sum(p);  o = alpha * o + p @ V_tile;  m = m_new
    A row whose tile is entirely masked skips the tile, so the first update
    never forms -inf - (-inf); alpha is 0 while m is still -inf
    [IO, "Executable recurrence, with an empty-state policy"]. After the last
    tile O = o / l (0 when l == 0) and lse = m + ln l (-inf when l == 0).
    """
    if isinstance(tile, bool) or not isinstance(tile, int) or tile < 1:
        raise ValueError(f"tile size {tile!r} is not an int of at least 1")
    q, k, v = _f64(q), _f64(k), _f64(v)
    Nq, Nk = q.shape[0], k.shape[0]
    rows = np.arange(Nq)
    keep_full = None if keep is None else np.broadcast_to(np.asarray(keep, dtype=bool), (Nq, Nk))
    m = np.full(Nq, NEG_INF)
    l = np.zeros(Nq)
    o = np.zeros((Nq, v.shape[1]))
    for start in range(0, Nk, tile):
        stop = min(start + tile, Nk)
        s = scale * (q @ k[start:stop].T)                          # [Nq, tile]
        # mask from the ABSOLUTE key positions start..stop-1, not tile-local ones
        j = np.arange(start, stop)[None, :]
        ok = np.ones((Nq, stop - start), dtype=bool)
        if causal:
            ok &= j <= (rows[:, None] + (Nk - Nq))
        if keep_full is not None:
            ok &= keep_full[:, start:stop]
        s = np.where(ok, s, NEG_INF)
        chunk_max = s.max(axis=1)
        live = ~np.isneginf(chunk_max)                 # rows with at least one allowed key here
        if not live.any():
            continue
        m_new = np.where(live, np.maximum(m, chunk_max), m)
        alpha = np.where(np.isneginf(m), 0.0, np.exp(np.where(live, m - m_new, 0.0)))
        alpha = np.where(live, alpha, 1.0)
        shift = np.where(live, m_new, 0.0)
        p = np.where(ok & live[:, None], np.exp(s - shift[:, None]), 0.0)
        l = alpha * l + p.sum(axis=1)
        o = alpha[:, None] * o + p @ v[start:stop]
        m = m_new
    has = l > 0
    safe_l = np.where(has, l, 1.0)
    out = np.where(has[:, None], o / safe_l[:, None], 0.0)
    lse = np.where(has, m + np.log(safe_l), NEG_INF)
    return out, lse


def online_attention(q, k, v, scale: float, causal: bool = False, keep=None,
                     tile: int = 128) -> Tuple[np.ndarray, np.ndarray]:
    """Batched ``online_attention_head`` over [B, H, N, d] inputs."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, _ = q.shape
    Nk = k.shape[2]
    out = np.zeros((B, H, Nq, v.shape[3]))
    lse = np.full((B, H, Nq), NEG_INF)
    kb = None if keep is None else np.broadcast_to(np.asarray(keep, dtype=bool), (B, H, Nq, Nk))
    for b in range(B):
        for h in range(H):
            out[b, h], lse[b, h] = online_attention_head(
                q[b, h], k[b, h], v[b, h], scale, causal,
                None if kb is None else kb[b, h], tile=tile)
    return out, lse


# ---------------------------------------------------------------------------
# Single-row forms, for the pages' worked examples
# ---------------------------------------------------------------------------

def _row_arrays(scores, values, tile):
    """One row's scores [N] and values [N] or [N, dv] as fp64 arrays (values
    as [N, dv]), after the input policy that [IO, "Executable recurrence,
    with an empty-state policy"] states: the counts must agree, the tile size
    is a positive int, a score is finite or -inf (a masked key; NaN and +inf
    are refused) and every value is finite. Anything else raises ValueError."""
    sc = np.asarray(scores, dtype=np.float64)
    vals = np.asarray(values, dtype=np.float64)
    if vals.ndim == 1:
        vals = vals.reshape(-1, 1)
    if sc.ndim != 1 or vals.ndim != 2 or len(sc) != len(vals):
        raise ValueError(f"{sc.shape} scores do not pair up with values of shape {vals.shape}")
    if isinstance(tile, bool) or not isinstance(tile, int) or tile < 1:
        raise ValueError(f"tile size {tile!r} is not an int of at least 1")
    if np.isnan(sc).any() or (sc == np.inf).any():
        raise ValueError("a score is NaN or +inf (allowed: finite, or -inf for a masked key)")
    if not np.isfinite(vals).all():
        raise ValueError("a value is NaN or infinite")
    return sc, vals


def online_row(scores, values, tile: int = 2, trace: bool = False):
    """One query row, new-max form [IO, "Keep only the state ..."; MEM, "Try it"].

    ``scores`` are already scaled and masked (-inf = masked); ``values`` is
    [N] or [N, dv]. The state after the keys folded in so far is the running
    max m of their visible scores, l = sum exp(s_j - m) and
    o = sum exp(s_j - m) v_j over them. Folding in one tile:
        m' = max(m, scores of the tile),  alpha = exp(m - m'),
        l' = alpha l + sum_tile w_j,  o' = alpha o + sum_tile w_j v_j,
    with w_j = exp(s_j - m') for visible keys and 0 for masked ones. Before
    any visible key m is -inf and l, o are 0; alpha is then taken as 0 (the
    empty state has nothing to rescale). The output is o / l, or zeros when l
    stays 0 (an empty or all-masked row). With ``trace=True`` the state
    (m, l, o, alpha) after each tile is returned too.
    """
    s, v = _row_arrays(scores, values, tile)
    visible = ~np.isneginf(s)
    m, l = NEG_INF, 0.0
    o = np.zeros(v.shape[1])
    states = []
    for t0 in range(0, len(s), tile):
        idx = slice(t0, min(len(s), t0 + tile))
        m_new = max(m, float(s[idx].max()))       # masked scores (-inf) never raise it
        alpha = math.exp(m - m_new) if np.isfinite(m) else 0.0
        base = m_new if np.isfinite(m_new) else 0.0
        w = np.where(visible[idx], np.exp(s[idx] - base), 0.0)
        l = alpha * l + float(w.sum())
        o = alpha * o + w @ v[idx]
        m = m_new
        states.append(dict(m=m, l=l, o=o.copy(), alpha=alpha))
    out = o / l if l > 0 else np.zeros_like(o)
    return (out, states) if trace else out


def blocklocal_row(scores, values, tile: int = 2, trace: bool = False):
    """One query row, block-local-max form [FAO, "The fix: tile the computation ..."].

    Each block is first reduced against its own max (m_block, l_block,
    acc_block); the running totals and the block are then both re-based to
    m_new with scale_old = exp(m_old - m_new) and scale_new =
    exp(m_block - m_new). Identical in exact arithmetic to ``online_row``.
    """
    s, v = _row_arrays(scores, values, tile)
    m, l = NEG_INF, 0.0
    acc = np.zeros(v.shape[1])
    states = []
    for start in range(0, s.shape[0], tile):
        bs = s[start:start + tile]
        m_block = bs.max()
        if np.isneginf(m_block):
            continue
        p = np.exp(bs - m_block)
        l_block = p.sum()
        acc_block = p @ v[start:start + tile]
        m_new = max(m, m_block)
        scale_old = 0.0 if np.isneginf(m) else math.exp(m - m_new)
        scale_new = math.exp(m_block - m_new)
        states.append(dict(m_block=m_block, l_block=l_block, acc_block=acc_block.copy(),
                           scale_old=scale_old, scale_new=scale_new))
        l = l * scale_old + l_block * scale_new
        acc = acc * scale_old + acc_block * scale_new
        m = m_new
        states[-1].update(m=m, l=l, acc=acc.copy())
    out = acc / l if l > 0 else np.zeros_like(acc)
    return (out, states) if trace else out


# ---------------------------------------------------------------------------
# Split-KV: partial (m, l, o) triples and their merge
# ---------------------------------------------------------------------------

def merge_partials(ms: Iterable[float], ls: Iterable[float],
                   os: Iterable[np.ndarray]) -> Tuple[np.ndarray, float]:
    """Merge per-split states into the exact result [NOTES, "Merging two blocks"].

    Each split s carries its own max m_s, its sum l_s of exp(score - m_s) and
    its unnormalised output o_s on the same base. Re-basing to the global max
    M = max_s m_s multiplies split s by exp(m_s - M) (one scalar per split);
    the re-based parts then add: L = sum l_s exp(m_s - M),
    O = sum o_s exp(m_s - M) / L, lse = M + ln L. Splits with l_s == 0 (empty
    or all masked) contribute nothing. No live split -> (0, -inf).
    """
    ms = np.asarray(list(ms), dtype=np.float64)
    ls = np.asarray(list(ls), dtype=np.float64)
    os = np.asarray([_f64(o) for o in os], dtype=np.float64)
    live = ls > 0
    if not live.any():
        return np.zeros(os.shape[1]), NEG_INF
    M = ms[live].max()
    w = np.where(live, np.exp(np.where(live, ms - M, 0.0)), 0.0)
    L = float((ls * w).sum())
    O = (w[:, None] * os).sum(axis=0) / L
    return O, M + math.log(L)


def splitkv_partials(q, k, v, scale: float, num_splits: int):
    """Per-split (m_s, l_s, o_s) for one query vector q [d] against k/v [Nk, d].

    Split s covers keys [s*c, min(Nk, (s+1)*c)) with c = ceil(Nk / num_splits)
    [MEM, "Where it helps, and where it does not": split the K/V sequence,
    then merge the partial results]. Each partial is the plain definition on
    its keys, left unnormalised.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Nk = k.shape[0]
    c = -(-Nk // num_splits) if Nk else 0
    ms, ls, os = [], [], []
    for s in range(num_splits):
        a, b = s * c, min(Nk, (s + 1) * c)
        if b <= a:
            ms.append(NEG_INF); ls.append(0.0); os.append(np.zeros(v.shape[1]))
            continue
        sc = scale * (k[a:b] @ q)
        m = sc.max()
        w = np.exp(sc - m)
        ms.append(m); ls.append(w.sum()); os.append(w @ v[a:b])
    return ms, ls, os


def splitkv_attention(q, k, v, scale: float, num_splits: int) -> Tuple[np.ndarray, np.ndarray]:
    """Decode (one query token per head) by split-KV partials + merge.

    q: [B, H, 1, d] (or [B, H, d]); k/v: [B, H, Nk, d]. Returns
    (O [B, H, 1, dv], lse [B, H, 1]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim == 3:
        q = q[:, :, None, :]
    B, H = q.shape[:2]
    out = np.zeros((B, H, 1, v.shape[3]))
    lse = np.full((B, H, 1), NEG_INF)
    for b in range(B):
        for h in range(H):
            parts = splitkv_partials(q[b, h, 0], k[b, h], v[b, h], scale, num_splits)
            out[b, h, 0], lse[b, h, 0] = merge_partials(*parts)
    return out, lse


__all__ = [
    "NEG_INF", "allowed_mask", "attend_head", "naive_attention",
    "online_attention_head", "online_attention", "online_row", "blocklocal_row",
    "merge_partials", "splitkv_partials", "splitkv_attention",
]
