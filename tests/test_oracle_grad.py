"""Pins of the fp64 backward oracle (CPU).

The oracle's gradient formulas are checked against things other than
themselves: central finite differences of the (separately pinned) forward
oracle, torch fp64 autograd through a plain softmax-attention written with
torch ops, and two invariants of the exact gradients. Planted mistakes in the
oracle's source must each fail at least one pin.
"""

import inspect
import types

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import attention_grad as AG

FUNCS = ["attend_head_grad", "attention_grad"]


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def pin_finite_differences(impl):
    """dL/dx by central differences of L = sum(O * G), O from the forward oracle."""
    for causal, keep_kind in [(False, None), (True, None), (True, "mask"), (False, "empty_row")]:
        Nq, Nk, d = 4, 6, 3
        q, k, v, g = _rand((Nq, d), 1), _rand((Nk, d), 2), _rand((Nk, d), 3), _rand((Nq, d), 4)
        keep = None
        if keep_kind == "mask":
            keep = _rand((Nq, Nk), 5) > -0.3
        elif keep_kind == "empty_row":
            keep = np.ones((Nq, Nk), dtype=bool)
            keep[1] = False
        scale = 0.7

        def loss(q_, k_, v_):
            o, _ = A.attend_head(q_, k_, v_, scale, causal, keep)
            return float((o * g).sum())

        dq, dk, dv = impl.attend_head_grad(q, k, v, g, scale, causal, keep)
        h = 1e-6
        for x, dx, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = [q, k, v]
                args_m = [q, k, v]
                args_p[which], args_m[which] = xp, xm
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert np.abs(num - dx).max() < 1e-7, (causal, keep_kind, which, np.abs(num - dx).max())


def pin_torch_autograd(impl):
    """torch fp64 autograd through softmax attention with a mask (no empty rows)."""
    for causal in (False, True):
        Nq, Nk, d, dv = 9, 11, 5, 4
        q, k, v, g = _rand((Nq, d), 11), _rand((Nk, d), 12), _rand((Nk, dv), 13), _rand((Nq, dv), 14)
        keep = _rand((Nq, Nk), 15) > -0.5
        keep[:, -1] = True      # every row keeps at least its last key (visible under bottom-right causal)
        scale = 0.45
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        s = scale * tq @ tk.T
        allowed = torch.tensor(keep)
        if causal:
            allowed &= torch.arange(Nk)[None, :] <= torch.arange(Nq)[:, None] + (Nk - Nq)
        s = s.masked_fill(~allowed, float("-inf"))
        o = torch.softmax(s, dim=-1) @ tv
        (o * torch.tensor(g)).sum().backward()
        dq, dk, dvv = impl.attend_head_grad(q, k, v, g, scale, causal, keep)
        for got, ref in ((dq, tq.grad), (dk, tk.grad), (dvv, tv.grad)):
            assert np.abs(got - ref.numpy()).max() < 1e-12


def pin_invariants(impl):
    """(1) Key gradients sum to zero: shifting every key by one vector moves a
    row's scores by a constant, which leaves O unchanged. (2) scale = 0: every
    allowed weight is uniform, so dq = dk = 0 and dv_j = sum over the rows i
    that see key j of do_i / (number of keys row i sees)."""
    for causal in (False, True):
        Nq, Nk, d = 7, 10, 4
        q, k, v, g = _rand((Nq, d), 21), _rand((Nk, d), 22), _rand((Nk, d), 23), _rand((Nq, d), 24)
        _, dk, _ = impl.attend_head_grad(q, k, v, g, 0.8, causal)
        assert np.abs(dk.sum(axis=0)).max() < 1e-12
        dq0, dk0, dv0 = impl.attend_head_grad(q, k, v, g, 0.0, causal)
        assert np.abs(dq0).max() == 0 and np.abs(dk0).max() == 0
        ok = A.allowed_mask(np.arange(Nq), Nk, Nq, causal, None)
        expect = np.zeros((Nk, d))
        for i in range(Nq):
            n = ok[i].sum()
            for j in np.nonzero(ok[i])[0]:
                expect[j] += g[i] / n
        assert np.abs(dv0 - expect).max() < 1e-12


def pin_batched(impl):
    """The batched form equals the per-head form on every (b, h)."""
    B, H, Nq, Nk, d = 2, 3, 5, 6, 4
    q, k, v, g = _rand((B, H, Nq, d), 31), _rand((B, H, Nk, d), 32), _rand((B, H, Nk, d), 33), _rand((B, H, Nq, d), 34)
    dq, dk, dv = impl.attention_grad(q, k, v, g, 0.5, True)
    for b in range(B):
        for h in range(H):
            r = impl.attend_head_grad(q[b, h], k[b, h], v[b, h], g[b, h], 0.5, True)
            for got, ref in zip((dq[b, h], dk[b, h], dv[b, h]), r):
                assert np.array_equal(got, ref)


PINS = [pin_finite_differences, pin_torch_autograd, pin_invariants, pin_batched]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(AG)


MUTANTS = [
    ("dS without the row term D", "dS = P * (dP - D[:, None])", "dS = P * dP"),
    ("D from dO not P", "D = (P * dP).sum(axis=1)", "D = dP.sum(axis=1)"),
    ("dq without scale", "dq[rb] = scale * (dS @ k)", "dq[rb] = (dS @ k)"),
    ("dq from v", "dq[rb] = scale * (dS @ k)", "dq[rb] = scale * (dS @ v)"),
    ("dk untransposed", "dk += scale * (dS.T @ q[rb])", "dk += scale * (P.T @ q[rb])"),
    ("dv from dS", "dv += P.T @ do[rb]", "dv += dS.T @ do[rb]"),
    ("dP transposed operand", "dP = do[rb] @ v.T", "dP = do[rb] @ k.T"),
    ("unnormalised P", "P = w / L[:, None]", "P = w"),
    ("mask ignored", "ok = allowed_mask(rb, Nk, Nq, causal, None if keep_full is None else keep_full[rb])",
     "ok = np.ones((rb.shape[0], Nk), dtype=bool)"),
]


def _mutant_impl(old, new):
    src = inspect.getsource(AG)
    assert src.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
    ns = {"__name__": "oracle_grad_mutant"}
    exec(compile(src.replace(old, new), "oracle_grad_mutant", "exec"), ns)
    return types.SimpleNamespace(**{f: ns[f] for f in FUNCS})


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    impl = _mutant_impl(old, new)
    caught = []
    for pin in PINS:
        try:
            pin(impl)
        except Exception:
            caught.append(pin.__name__)
    assert caught, f"planted mistake '{name}' passed every pin"
