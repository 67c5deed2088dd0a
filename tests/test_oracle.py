"""Pins for the fp64 oracle (CPU only).

Each ``pin_*`` checks the oracle against something other than itself: values
the pages print for worked examples (tests/golden/worked_examples.json), a
library routine (torch's fp64 scaled_dot_product_attention,
scipy.special.logsumexp / expit), closed forms, invariants of the exact
result, and brute force in pure Python over every mask of tiny rows.

The mutation tests at the bottom plant plausible mistakes in a copy of the
oracle module (a dropped term, a wrong sign, a tile-local causal index, a
transposed or wrong operand) and require at least one pin to reject each.
"""

import inspect
import itertools
import json
import math
import os
import types

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

from oracle import attention as A

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))

HAND = GOLDEN["hand_rel_tol"]

FUNCS = ["attend_head", "online_attention_head", "online_row", "blocklocal_row",
         "merge_partials", "splitkv_partials", "splitkv_attention", "allowed_mask"]


def real_impl():
    return types.SimpleNamespace(**{f: getattr(A, f) for f in FUNCS})


def printed(x, spec, what="", rel=0.0):
    """x rounds to the value the page prints with ``decimals`` decimals (``rel``
    widens this for intermediates the page computed from rounded factors)."""
    vals = np.atleast_1d(np.asarray(spec["value"], dtype=np.float64))
    tol = 0.5 * 10.0 ** (-spec["decimals"]) + 1e-12 + rel * np.abs(vals)
    x = np.atleast_1d(np.asarray(x, dtype=np.float64))
    assert x.shape == vals.shape, what
    assert np.all(np.abs(x - vals) <= tol), f"{what}: {x} vs printed {vals} (tol {tol})"


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_worked_examples(impl):
    for ex in GOLDEN["examples"]:
        s = np.array(ex["scores"])
        v = np.array(ex["values"])
        t = ex["tile"]
        out, st = impl.online_row(s, v, t, trace=True)
        printed(out[0], ex["output"], ex["name"] + " online_row")
        if "output_long" in ex:
            printed(out[0], ex["output_long"], ex["name"] + " online_row long")
        outb, stb = impl.blocklocal_row(s, v, t, trace=True)
        printed(outb[0], ex["output"], ex["name"] + " blocklocal_row")
        for i, step in enumerate(ex.get("blocklocal_steps", [])):
            got = stb[i]
            assert got["m_block"] == step["m_block"] and got["m"] == step["m"]
            for key in ("l_block", "acc_block", "scale_old", "scale_new", "l", "acc"):
                if key in step:
                    printed(np.ravel(got[key])[0], step[key], f"{ex['name']} step{i} {key}", HAND)
            # the new-max form holds the same running (m, l, o) after every tile
            printed(st[i]["l"], step["l"], f"{ex['name']} new-max step{i} l", HAND)
            printed(st[i]["o"][0], step["acc"], f"{ex['name']} new-max step{i} o", HAND)
        for i, step in enumerate(ex.get("newmax_steps", [])):
            got = st[i]
            assert abs(got["m"] - step["m"]) < 1e-15
            for key in ("alpha", "l", "o"):
                if key in step:
                    printed(np.ravel(got[key])[0], step[key], f"{ex['name']} step{i} {key}", HAND)
        # the batched paths, with q = [1], k_j = [s_j], scale 1 so that score_j = s_j
        q1 = np.array([[1.0]])
        kk = s[:, None]
        vv = v[:, None]
        o, lse = impl.attend_head(q1, kk, vv, 1.0)
        printed(o[0, 0], ex["output"], ex["name"] + " attend_head")
        assert abs(lse[0] - scipy.special.logsumexp(s)) < 1e-12
        o2, lse2 = impl.online_attention_head(q1, kk, vv, 1.0, tile=t)
        printed(o2[0, 0], ex["output"], ex["name"] + " online_attention_head")
        assert abs(lse2[0] - scipy.special.logsumexp(s)) < 1e-12
        if "direct_weights" in ex:
            printed(np.exp(s - lse[0]), ex["direct_weights"], "direct weights", HAND)
            printed(np.exp(lse[0] - s.max()), ex["direct_sum"], "direct sum", HAND)


def _sdpa(q, k, v, scale, causal=False, mask=None):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    return F.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=m, is_causal=causal,
                                          scale=scale)[0, 0].numpy()


def pin_library(impl):
    rng = np.random.default_rng(7)
    for (Nq, Nk, d, dv) in [(5, 7, 4, 3), (16, 16, 8, 8), (33, 17, 16, 5), (9, 9, 3, 6)]:
        q = rng.standard_normal((Nq, d))
        k = rng.standard_normal((Nk, d))
        v = rng.standard_normal((Nk, dv))
        cases = [(False, None)]
        if Nq == Nk:
            cases.append((True, None))
        keep = rng.random((Nq, Nk)) < 0.5
        keep[np.arange(Nq), rng.integers(0, Nk, Nq)] = True   # no empty rows here
        cases.append((False, keep))
        # a negative scale is a valid input of softmax(scale q k^T): the weights
        # then favour the smallest dot products
        for (causal, mask), scale in itertools.product(cases, (0.37, -0.6)):
            raw = scale * (q @ k.T)
            # torch's fp64 path takes the square root of its scale, so the
            # negative case asks it for |scale| (q . -k) = scale (q . k), exactly
            ref = _sdpa(q, np.sign(scale) * k, v, abs(scale), causal, mask)
            allowed = np.ones((Nq, Nk), bool) if mask is None else mask.copy()
            if causal:
                allowed &= np.tril(np.ones((Nq, Nk), bool))
            ref_lse = scipy.special.logsumexp(np.where(allowed, raw, -np.inf), axis=1)
            for fn in (lambda: impl.attend_head(q, k, v, scale, causal, mask),
                       lambda: impl.online_attention_head(q, k, v, scale, causal, mask, tile=3),
                       lambda: impl.online_attention_head(q, k, v, scale, causal, mask, tile=16)):
                o, lse = fn()
                assert np.abs(o - ref).max() < 1e-12
                assert np.abs(lse - ref_lse).max() < 1e-12


def pin_try_it(impl):
    cfg = GOLDEN["tiled_vs_library"]
    torch.manual_seed(cfg["seed"])
    q, k, v = (torch.randn(cfg["N"], cfg["d"], dtype=torch.float64) for _ in range(3))
    ref = F.scaled_dot_product_attention(q[None, None], k[None, None], v[None, None])[0, 0].numpy()
    scale = 1.0 / math.sqrt(cfg["d"])
    o, _ = impl.online_attention_head(q.numpy(), k.numpy(), v.numpy(), scale, tile=cfg["block"])
    # the page prints ~6e-16; allow for a different BLAS summation order
    assert np.abs(o - ref).max() < 1e-14
    o2, _ = impl.attend_head(q.numpy(), k.numpy(), v.numpy(), scale)
    assert np.abs(o2 - ref).max() < 1e-14


def _brute(q, k, v, scale, causal, keep):
    """Pure-Python loops: the definition, one row at a time."""
    Nq, Nk = len(q), len(k)
    outs, lses = [], []
    for i in range(Nq):
        allowed = [j for j in range(Nk)
                   if (not causal or j <= i + (Nk - Nq)) and (keep is None or keep[i][j])]
        if not allowed:
            outs.append([0.0] * len(v[0]) if Nk else [0.0])
            lses.append(-math.inf)
            continue
        s = {j: scale * sum(a * b for a, b in zip(q[i], k[j])) for j in allowed}
        M = max(s.values())
        w = {j: math.exp(s[j] - M) for j in allowed}
        L = sum(w.values())
        outs.append([sum(w[j] * v[j][c] for j in allowed) / L for c in range(len(v[0]))])
        lses.append(M + math.log(L))
    return outs, lses


def pin_bruteforce(impl):
    rng = np.random.default_rng(11)
    for Nq in (1, 2, 3):
        for Nk in (1, 2, 3, 4):
            q = rng.standard_normal((Nq, 2))
            k = rng.standard_normal((Nk, 2))
            v = rng.standard_normal((Nk, 3))
            for bits in range(2 ** Nk):
                row = [(bits >> j) & 1 == 1 for j in range(Nk)]
                keep = np.array([row] * Nq)
                for causal in (False, True):
                    ro, rl = _brute(q.tolist(), k.tolist(), v.tolist(), 0.9, causal, keep.tolist())
                    ro, rl = np.array(ro), np.array(rl)
                    for fn in (lambda: impl.attend_head(q, k, v, 0.9, causal, keep),
                               lambda: impl.online_attention_head(q, k, v, 0.9, causal, keep, tile=1),
                               lambda: impl.online_attention_head(q, k, v, 0.9, causal, keep, tile=2)):
                        o, l = fn()
                        assert np.abs(o - ro).max() < 1e-12, (Nq, Nk, bits, causal)
                        assert np.array_equal(np.isneginf(l), np.isneginf(rl))
                        fin = np.isfinite(rl)
                        assert np.abs(l[fin] - rl[fin]).max(initial=0) < 1e-12


def pin_closed_forms(impl):
    rng = np.random.default_rng(3)
    d = 6
    q = rng.standard_normal((4, d))
    # one key: output is that key's value, lse its score
    k1 = rng.standard_normal((1, d))
    v1 = rng.standard_normal((1, 5))
    for fn in (impl.attend_head, lambda *a: impl.online_attention_head(*a, tile=2)):
        o, lse = fn(q, k1, v1, 0.5)
        assert np.abs(o - v1[0]).max() < 1e-14
        assert np.abs(lse - 0.5 * (q @ k1[0])).max() < 1e-14
    # uniform scores (q = 0): plain mean of V, lse = ln Nk
    k = rng.standard_normal((10, d))
    v = rng.standard_normal((10, 5))
    for fn in (impl.attend_head, lambda *a: impl.online_attention_head(*a, tile=3)):
        o, lse = fn(np.zeros((3, d)), k, v, 0.7)
        assert np.abs(o - v.mean(axis=0)).max() < 1e-14
        assert np.abs(lse - math.log(10)).max() < 1e-14
    # two keys: O = v0 + (v1 - v0) * expit(s1 - s0), lse = logaddexp(s0, s1)
    k2 = rng.standard_normal((2, d))
    v2 = rng.standard_normal((2, 4))
    s = 0.8 * (q @ k2.T)
    exp_o = v2[0] + (v2[1] - v2[0]) * scipy.special.expit(s[:, 1] - s[:, 0])[:, None]
    for fn in (impl.attend_head, lambda *a: impl.online_attention_head(*a, tile=1)):
        o, lse = fn(q, k2, v2, 0.8)
        assert np.abs(o - exp_o).max() < 1e-13
        assert np.abs(lse - np.logaddexp(s[:, 0], s[:, 1])).max() < 1e-13
    # causal, square: row 0 sees only key 0
    kq = rng.standard_normal((4, d))
    vq = rng.standard_normal((4, 3))
    for fn in (impl.attend_head, lambda *a: impl.online_attention_head(*a, tile=2)):
        o, lse = fn(q, kq, vq, 0.5, True)
        assert np.abs(o[0] - vq[0]).max() < 1e-14
        assert abs(lse[0] - 0.5 * q[0] @ kq[0]) < 1e-14
    # causal with Nq > Nk (bottom-right): rows i < Nq - Nk see nothing, row Nq - Nk sees key 0
    k2c = rng.standard_normal((2, d))
    v2c = rng.standard_normal((2, 3))
    for fn in (impl.attend_head, lambda *a: impl.online_attention_head(*a, tile=1)):
        o, lse = fn(q, k2c, v2c, 0.5, True)
        assert np.all(o[:2] == 0) and np.all(np.isneginf(lse[:2]))
        assert np.abs(o[2] - v2c[0]).max() < 1e-14
        assert np.all(np.isfinite(lse[2:]))
    # causal with Nq < Nk: the last query row sees every key, so it equals non-causal
    kl = rng.standard_normal((7, d))
    vl = rng.standard_normal((7, 3))
    oc, lc = impl.attend_head(q[:2], kl, vl, 0.5, True)
    on, ln_ = impl.attend_head(q[:2], kl, vl, 0.5, False)
    assert np.abs(oc[1] - on[1]).max() < 1e-14 and abs(lc[1] - ln_[1]) < 1e-14
    assert not np.allclose(oc[0], on[0])
    # no keys at all, and a fully masked row: zeros and -inf
    o, lse = impl.attend_head(q, np.zeros((0, d)), np.zeros((0, 3)), 0.5)
    assert o.shape == (4, 3) and np.all(o == 0) and np.all(np.isneginf(lse))
    keep = np.ones((4, 10), bool)
    keep[2] = False
    for fn in (impl.attend_head, lambda *a: impl.online_attention_head(*a, tile=4)):
        o, lse = fn(q, k, v, 0.5, False, keep)
        assert np.all(o[2] == 0) and np.isneginf(lse[2]) and np.all(np.isfinite(lse[[0, 1, 3]]))
    assert np.all(impl.online_row([-np.inf, -np.inf, -np.inf], np.ones((3, 2)), 2) == 0)
    assert np.all(impl.online_row([], np.zeros((0, 2)), 2) == 0)


def pin_invariants(impl):
    rng = np.random.default_rng(5)
    q = rng.standard_normal((6, 5))
    k = rng.standard_normal((9, 5))
    v = rng.standard_normal((9, 4))
    k[:, -1] = 1.0
    scale = 0.25
    o0, l0 = impl.attend_head(q, k, v, scale)
    for c in (1e3, -1e3):
        q2 = q.copy()
        q2[:, -1] += c / scale            # every score of every row moves by exactly c
        for fn in (impl.attend_head, lambda *a: impl.online_attention_head(*a, tile=4)):
            o, l = fn(q2, k, v, scale)
            assert np.abs(o - o0).max() < 1e-10
            assert np.abs(l - (l0 + c)).max() < 1e-9
    # different rows shifted by different large constants (+1e3, -1e3, 0, ...):
    # each row's result is still unchanged, so the max must be per row
    offs = np.array([1e3, -1e3, 0.0, 5e2, -7e2, 1e3])
    q3 = q.copy()
    q3[:, -1] += offs / scale
    for fn in (impl.attend_head, lambda *a: impl.online_attention_head(*a, tile=4)):
        o, l = fn(q3, k, v, scale)
        assert np.abs(o - o0).max() < 1e-10
        assert np.abs(l - (l0 + offs)).max() < 1e-9
    # permuting keys (with their values) changes nothing when not causal
    perm = rng.permutation(9)
    for fn in (impl.attend_head, lambda *a: impl.online_attention_head(*a, tile=2)):
        o, l = fn(q, k[perm], v[perm], scale)
        assert np.abs(o - o0).max() < 1e-13 and np.abs(l - l0).max() < 1e-13
    # linear in V
    v2 = rng.standard_normal((9, 4))
    oa, _ = impl.attend_head(q, k, v, scale)
    ob, _ = impl.attend_head(q, k, v2, scale)
    oc, _ = impl.attend_head(q, k, 2.0 * v - 3.0 * v2, scale)
    assert np.abs(oc - (2.0 * oa - 3.0 * ob)).max() < 1e-12
    # rows are independent: a subset of rows gives the same rows
    sub = np.array([4, 1])
    os_, ls_ = impl.attend_head(q, k, v, scale, rows=sub)
    assert np.abs(os_ - o0[sub]).max() < 1e-15 and np.abs(ls_ - l0[sub]).max() < 1e-15


def pin_merge(impl):
    # the toy example as two one-key splits: m = (0, ln 2), l = (1, 1), o = (10, 20)
    O, lse = impl.merge_partials([0.0, math.log(2)], [1.0, 1.0], [np.array([10.0]), np.array([20.0])])
    assert abs(O[0] - 50.0 / 3.0) < 1e-12 and abs(lse - math.log(3)) < 1e-12
    # an empty split contributes nothing; no live split -> (0, -inf)
    O, lse = impl.merge_partials([-np.inf, 1.5], [0.0, 2.0], [np.zeros(2), np.array([4.0, 6.0])])
    assert np.abs(O - np.array([2.0, 3.0])).max() < 1e-15 and abs(lse - (1.5 + math.log(2))) < 1e-15
    O, lse = impl.merge_partials([-np.inf], [0.0], [np.zeros(3)])
    assert np.all(O == 0) and np.isneginf(lse)
    rng = np.random.default_rng(9)
    for Nk in (1, 7, 64):
        q = rng.standard_normal((2, 3, 1, 8))
        k = rng.standard_normal((2, 3, Nk, 8))
        v = rng.standard_normal((2, 3, Nk, 8))
        for splits in (1, 3, 16, 100):
            o, l = impl.splitkv_attention(q, k, v, 0.3, splits)
            for b in range(2):
                for h in range(3):
                    ro = _sdpa(q[b, h], k[b, h], v[b, h], 0.3)
                    rl = scipy.special.logsumexp(0.3 * (k[b, h] @ q[b, h, 0]))
                    assert np.abs(o[b, h] - ro).max() < 1e-13
                    assert abs(l[b, h, 0] - rl) < 1e-13


PINS = [pin_worked_examples, pin_library, pin_try_it, pin_bruteforce,
        pin_closed_forms, pin_invariants, pin_merge]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(real_impl())


def test_input_checks():
    """The executable recurrence rejects NaN / +inf scores, non-finite values, bad tiles."""
    with pytest.raises(ValueError):
        A.online_row([1.0, np.nan], [1.0, 2.0])
    with pytest.raises(ValueError):
        A.online_row([1.0, np.inf], [1.0, 2.0])
    with pytest.raises(ValueError):
        A.online_row([1.0, 2.0], [1.0, np.inf])
    with pytest.raises(ValueError):
        A.online_row([1.0, 2.0], [1.0, 2.0], tile=0)
    with pytest.raises(ValueError):
        A.online_row([1.0, 2.0], [1.0, 2.0], tile=1.5)
    with pytest.raises(ValueError):
        A.online_row([1.0, 2.0, 3.0], [1.0, 2.0])
    with pytest.raises(ValueError):
        A.online_attention_head(np.ones((2, 2)), np.ones((2, 2)), np.ones((2, 2)), 1.0, tile=0)
    assert np.isfinite(A.online_row([1.0, -np.inf], [1.0, 2.0])).all()


def test_batched_matches_heads():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((2, 2, 5, 4))
    k = rng.standard_normal((2, 2, 7, 4))
    v = rng.standard_normal((2, 2, 7, 3))
    keep = rng.random((2, 2, 1, 7)) < 0.7
    for causal in (False, True):
        o, l = A.naive_attention(q, k, v, 0.5, causal, keep)
        o2, l2 = A.online_attention(q, k, v, 0.5, causal, keep, tile=3)
        for b in range(2):
            for h in range(2):
                ro, rl = _brute(q[b, h].tolist(), k[b, h].tolist(), v[b, h].tolist(), 0.5, causal,
                                np.broadcast_to(keep[b, h], (5, 7)).tolist())
                assert np.abs(o[b, h] - np.array(ro)).max() < 1e-12
                assert np.abs(o2[b, h] - np.array(ro)).max() < 1e-12
                fin = np.isfinite(rl)
                assert np.array_equal(np.isfinite(l[b, h]), fin)
                assert np.abs(l[b, h][fin] - np.array(rl)[fin]).max(initial=0) < 1e-12


def test_byte_arithmetic_fixture():
    """The FLOP and byte accounting used by the benchmark matches the page's worked numbers."""
    from io_aware_exact_fa_gb300.workloads import Workload
    ba = GOLDEN["byte_arithmetic"]
    w = Workload("one_head", 1, 1, ba["N"], ba["N"], ba["d"], 1.0)
    printed(w.flops(False) / 1e9, ba["matmul_flops_gflop"], "4 N^2 d")
    qkvo = 4 * ba["N"] * ba["d"] * 2
    assert qkvo == ba["min_io_bytes"]
    assert w.io_bytes() - 4 * ba["N"] == ba["min_io_bytes"]      # minus the fp32 lse we add
    assert qkvo + 4 * ba["N"] ** 2 * 2 == ba["materializing_total_bytes"]


# ---------------------------------------------------------------------------
# mutation tests: every planted mistake must be caught by some pin
# ---------------------------------------------------------------------------

MUTANTS = [
    ("no max subtraction", "w = np.where(ok, np.exp(s - M[:, None]), 0.0)",
     "w = np.where(ok, np.exp(s), 0.0)"),
    ("lse drops the max", "np.where(any_ok, M + np.log(safe_L), NEG_INF)",
     "np.where(any_ok, np.log(safe_L), NEG_INF)"),
    ("scale dropped", "s = scale * (q[rb] @ k.T)", "s = (q[rb] @ k.T)"),
    ("causal off by one", "allowed &= j <= (rows[:, None] + (Nk - Nq))",
     "allowed &= j < (rows[:, None] + (Nk - Nq))"),
    ("causal alignment sign", "allowed &= j <= (rows[:, None] + (Nk - Nq))",
     "allowed &= j <= (rows[:, None] + (Nq - Nk))"),
    ("wrong operand (k for v)", "num = w @ v", "num = w @ k"),
    ("online: l not rescaled", "l = alpha * l + p.sum(axis=1)", "l = l + p.sum(axis=1)"),
    ("online: o not rescaled", "o = alpha[:, None] * o + p @ v[start:stop]", "o = o + p @ v[start:stop]"),
    ("online: tile-local causal index", "ok &= j <= (rows[:, None] + (Nk - Nq))",
     "ok &= (j - start) <= (rows[:, None] + (Nk - Nq))"),
    ("online: alpha sign", "alpha = np.where(np.isneginf(m), 0.0, np.exp(np.where(live, m - m_new, 0.0)))",
     "alpha = np.where(np.isneginf(m), 0.0, np.exp(np.where(live, m_new - m, 0.0)))"),
    ("row: alpha sign", "alpha = math.exp(m - m_new) if np.isfinite(m) else 0.0",
     "alpha = math.exp(m_new - m) if np.isfinite(m) else 0.0"),
    ("row: dropped alpha on o", "o = alpha * o + w @ v[idx]", "o = o + w @ v[idx]"),
    ("row: masked keys weighted", "w = np.where(visible[idx], np.exp(s[idx] - base), 0.0)",
     "w = np.exp(np.where(visible[idx], s[idx], 0.0) - base)"),
    ("blocklocal: scale_new dropped", "scale_new = math.exp(m_block - m_new)", "scale_new = 1.0"),
    ("merge: weight sign", "w = np.where(live, np.exp(np.where(live, ms - M, 0.0)), 0.0)",
     "w = np.where(live, np.exp(np.where(live, M - ms, 0.0)), 0.0)"),
    ("merge: unweighted sum", "O = (w[:, None] * os).sum(axis=0) / L", "O = os.sum(axis=0) / L"),
    ("split: tail keys dropped", "c = -(-Nk // num_splits) if Nk else 0", "c = Nk // num_splits if Nk else 0"),
    ("row max over wrong axis", "M = np.where(any_ok, s.max(axis=1), 0.0)",
     "M = np.where(any_ok, s.max(), 0.0)"),
]


def _mutant_impl(old, new):
    src = inspect.getsource(A)
    assert src.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
    ns = {"__name__": "oracle_mutant"}
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), ns)
    return types.SimpleNamespace(**{f: ns[f] for f in FUNCS})


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    impl = _mutant_impl(old, new)
    caught = []
    for pin in PINS:
        try:
            pin(impl)
        except Exception:   # an AssertionError or a crash both reject the mutant
            caught.append(pin.__name__)
    assert caught, f"planted mistake '{name}' passed every pin"
