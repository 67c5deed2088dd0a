"""Parity helpers: compare CUDA outputs with the fp64 oracle on the same bytes.

Tolerances (bf16 inputs, fp32 accumulation): max |dO| <= 1e-2,
mean |dO| <= 1e-3, |d lse| <= 1e-3 on finite lse; rows the oracle gives
lse = -inf must come back with lse = -inf and O = 0 exactly.

O is returned in bf16, and rounding the exact result to bf16 alone moves an
element by up to half a bf16 ulp (2^-6 for |O| in [4, 8)), which exceeds
1e-2 wherever |O| >= 2.56. The 1e-2 bound is read as the error of the
computation before that final rounding: each element may differ from the
oracle by 1e-2 plus half a bf16 ulp of the oracle's value.
"""

import numpy as np
import torch

from oracle import attention as A

TOL_MAX = 1e-2
TOL_MEAN = 1e-3
TOL_LSE = 1e-3


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_heads(q, k, v, scale, causal, keep=None, rows=None, heads=None):
    """Oracle for selected (b, h) and rows. q/k/v: CPU bf16 tensors [B,H,N,d].

    ``keep``: bool tensor broadcastable to [B,H,Nq,Nk] or None. ``rows``:
    None (all rows) or a 1-D index array. ``heads``: list of (b, h) or None
    (all). Returns {(b, h): (O [r, d], lse [r])}.
    """
    B, H, Nq, _ = q.shape
    Nk = k.shape[2]
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    kb = None
    if keep is not None:
        kb = keep.expand(B, H, keep.shape[2], Nk)
    out = {}
    for b, h in heads:
        kh = None
        if kb is not None:
            kh = kb[b, h].numpy()
            if kh.shape[0] == 1:
                kh = np.broadcast_to(kh, (Nq, Nk))
        out[(b, h)] = A.attend_head(to64(q[b, h]), to64(k[b, h]), to64(v[b, h]), scale, causal, kh,
                                    rows=None if rows is None else np.asarray(rows))
    return out


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half the bf16 spacing at |x| (8 significant bits): 2^(floor(log2|x|) - 8).
    Zero below the smallest normal number."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    out = np.zeros_like(a)
    nz = a >= 2.0 ** -126
    out[nz] = np.exp2(np.floor(np.log2(a[nz])) - 8.0)
    return out


def compare(o_gpu: np.ndarray, lse_gpu: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray, what: str = ""):
    """Element-wise comparison with the stated tolerances; returns stats."""
    assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    d = np.abs(o_gpu - o_ref)
    mx, mean = float(d.max(initial=0.0)), float(d.mean()) if d.size else 0.0
    excess = float((d - half_ulp_bf16(o_ref)).max(initial=0.0))  # error beyond the output rounding
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), empty), f"{what}: -inf lse rows differ"
    assert np.all(o_gpu[empty] == 0), f"{what}: an all-masked row is not exactly zero"
    fin = ~empty
    dl = float(np.abs(lse_gpu[fin] - lse_ref[fin]).max(initial=0.0))
    assert excess <= TOL_MAX, f"{what}: max |dO| = {mx:.3e}, {excess:.3e} beyond bf16 output rounding > {TOL_MAX}"
    assert mean <= TOL_MEAN, f"{what}: mean |dO| = {mean:.3e} > {TOL_MEAN}"
    assert dl <= TOL_LSE, f"{what}: max |dlse| = {dl:.3e} > {TOL_LSE}"
    return dict(max_abs=mx, max_beyond_rounding=excess, mean_abs=mean, max_lse=dl)
