"""Pins of the decode-variants oracle (CPU).

The oracle composes the pinned forward definition per (b, h); these pins check
the composition -- the K/V head each query head reads, the cut to the
sequence's length, and the causal rule among the new tokens -- against code
that shares none of it: torch fp64 with K/V heads expanded by
repeat_interleave and a visibility mask built element by element from the
rule "token t of sequence b sees key j iff j < L_b and j <= L_b - Nq + t",
and pure-Python brute force on tiny inputs. Planted mistakes must each fail
a pin.
"""

import inspect
import math
import types

import numpy as np
import pytest
import torch

from oracle import decode_variants as DV


def _case(seed, B=3, H=6, Hkv=2, Nq=3, Nk=11, d=4):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, Nq, d))
    k = rng.standard_normal((B, Hkv, Nk, d))
    v = rng.standard_normal((B, Hkv, Nk, d))
    return q, k, v


def pin_torch_mask(impl):
    """torch fp64 reference with an explicit element-wise visibility mask."""
    for seed, lens in ((1, [11, 5, 2]), (2, [0, 7, 11]), (3, [3, 1, 9])):
        q, k, v = _case(seed)
        B, H, Nq, d = q.shape
        Hkv, Nk = k.shape[1], k.shape[2]
        G = H // Hkv
        scale = 0.6
        tq, tk, tv = (torch.tensor(x) for x in (q, k, v))
        tk, tv = tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1)  # [B, H, Nk, d]
        allowed = torch.zeros(B, H, Nq, Nk, dtype=torch.bool)
        for b in range(B):
            for t in range(Nq):
                for j in range(Nk):
                    allowed[b, :, t, j] = j < lens[b] and j <= lens[b] - Nq + t
        s = scale * tq @ tk.transpose(-1, -2)
        s = s.masked_fill(~allowed, float("-inf"))
        lse_ref = torch.logsumexp(s, dim=-1)
        p = torch.softmax(s, dim=-1).nan_to_num(0.0)  # rows without a visible key -> 0
        o_ref = p @ tv
        o, lse = impl.decode_grouped_attention(q, k, v, lens, scale)
        assert np.abs(o - o_ref.numpy()).max() < 1e-12
        none = ~allowed.any(-1).numpy()
        assert np.all(np.isneginf(lse[none])) and np.all(np.isneginf(lse_ref.numpy()[none]))
        assert np.abs(lse[~none] - lse_ref.numpy()[~none]).max() < 1e-12
        assert none.any(), "the cases include tokens that see no key"


def pin_brute_force(impl):
    """Pure-Python loops on a tiny case: visible keys, weights, weighted sum."""
    q, k, v = _case(7, B=2, H=4, Hkv=2, Nq=2, Nk=5, d=2)
    lens = [4, 1]
    scale = 1.3
    o, lse = impl.decode_grouped_attention(q, k, v, lens, scale)
    for b in range(2):
        for h in range(4):
            kv = h // 2
            for t in range(2):
                vis = [j for j in range(5) if j < lens[b] and j <= lens[b] - 2 + t]
                if not vis:
                    assert np.all(o[b, h, t] == 0) and lse[b, h, t] == -math.inf
                    continue
                sc = [scale * sum(q[b, h, t, c] * k[b, kv, j, c] for c in range(2)) for j in vis]
                mx = max(sc)
                w = [math.exp(x - mx) for x in sc]
                tot = sum(w)
                for c in range(2):
                    ref = sum(wi * v[b, kv, j, c] for wi, j in zip(w, vis)) / tot
                    assert abs(o[b, h, t, c] - ref) < 1e-12
                assert abs(lse[b, h, t] - (mx + math.log(tot))) < 1e-12


def pin_defaults(impl):
    """No lengths means every key of the cache; one token sees them all."""
    q, k, v = _case(11, Nq=1)
    o1, l1 = impl.decode_grouped_attention(q, k, v, None, 0.5)
    o2, l2 = impl.decode_grouped_attention(q, k, v, [k.shape[2]] * q.shape[0], 0.5)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # token 0 of 1 sees keys 0 .. L-1: the plain softmax over the whole prefix
    b, h = 1, 5
    s = 0.5 * k[b, h // 3] @ q[b, h, 0]
    w = np.exp(s - s.max())
    assert np.abs(o1[b, h, 0] - (w / w.sum()) @ v[b, h // 3]).max() < 1e-12


PINS = [pin_torch_mask, pin_brute_force, pin_defaults]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(DV)


MUTANTS = [
    ("K/V head by modulo", "g = h // G", "g = h % Hkv"),
    ("lengths ignored", "L = Nk if seqlens is None else min(max(int(seqlens[b]), 0), Nk)", "L = Nk"),
    ("new tokens not causal", "causal=True)", "causal=False)"),
    ("whole cache instead of the prefix", "_f64(k[b, g, :L]), _f64(v[b, g, :L])", "_f64(k[b, g]), _f64(v[b, g])"),
    ("length off by one", "_f64(k[b, g, :L]), _f64(v[b, g, :L])",
     "_f64(k[b, g, :max(L - 1, 0)]), _f64(v[b, g, :max(L - 1, 0)])"),
]


def _mutant(old, new):
    src = inspect.getsource(DV)
    assert src.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
    ns = {"__name__": "decode_variants_mutant"}
    exec(compile(src.replace(old, new), "decode_variants_mutant", "exec"), ns)
    return types.SimpleNamespace(decode_grouped_attention=ns["decode_grouped_attention"])


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    impl = _mutant(old, new)
    caught = []
    for pin in PINS:
        try:
            pin(impl)
        except Exception:
            caught.append(pin.__name__)
    assert caught, f"planted mistake '{name}' passed every pin"
