"""Pins for the FP8 oracle (oracle/fp8.py), CPU only.

Each pin checks the oracle against something other than itself: torch's
float8_e4m3fn conversion (a library routine) over all 256 codes, values the
e4m3 format definition fixes, torch's fp64 scaled_dot_product_attention on
the decoded inputs, and invariants of the descale factors. The mutation
tests plant plausible mistakes (a wrong exponent bias, subnormals decoded as
normals, a dropped sign, a descale on the wrong operand) in a copy of the
module and require some pin to fail.
"""

import inspect
import math
import types

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from io_aware_exact_fa_gb300 import workloads as W
from oracle import fp8 as FP8


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_decode_library(m):
    codes = np.arange(256)
    got, ref = m.e4m3_decode(codes), _torch_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))


def pin_decode_format_values(m):
    # values the format fixes: 1 = 0x38 (exponent field 7 = bias), 448 = 0x7E
    # (largest finite), 2^-9 = 0x01 (smallest subnormal), 2^-6 = 0x08
    # (smallest normal), 0x07 = 7/8 * 2^-6 (largest subnormal), 0xB8 = -1,
    # 0x7F and 0xFF NaN (no infinities)
    d = m.e4m3_decode(np.array([0x38, 0x7E, 0x01, 0x08, 0x07, 0xB8, 0x7F, 0xFF, 0x00, 0x3C]))
    assert d[0] == 1.0 and d[1] == 448.0 and d[2] == 2.0 ** -9 and d[3] == 2.0 ** -6
    assert d[4] == 7 / 8 * 2.0 ** -6 and d[5] == -1.0
    assert np.isnan(d[6]) and np.isnan(d[7]) and d[8] == 0.0 and d[9] == 1.5


def _inputs(seed, Nq, Nk, d, dv=None):
    (q8, k8, v8), ds = W.make_qkv_fp8(1, 1, Nq, Nk, d, seed=seed)
    if dv is not None:
        v8 = v8[..., :dv]
    return q8[0, 0].numpy(), k8[0, 0].numpy(), v8[0, 0].numpy(), ds


def pin_attention_library(m):
    for (Nq, Nk, d, causal, scale) in [(9, 13, 16, False, 0.25), (16, 16, 32, True, 0.125),
                                       (5, 40, 8, False, -0.3)]:
        q8, k8, v8, (dq, dk, dv) = _inputs(Nq * 7 + Nk, Nq, Nk, d)
        o, lse = m.attend_head_fp8(q8, k8, v8, dq, dk, dv, scale, causal)
        qf, kf, vf = _torch_decode(q8) * dq, _torch_decode(k8) * dk, _torch_decode(v8) * dv
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None, None]
        # torch's fp64 path takes the square root of its scale: ask it for
        # |scale| with the keys negated when scale < 0 (an exact identity)
        ref = F.scaled_dot_product_attention(t(qf), t(np.sign(scale) * kf), t(vf), is_causal=causal,
                                             scale=abs(scale))[0, 0].numpy()
        assert np.abs(o - ref).max() < 1e-12
        s = scale * (qf @ kf.T)
        if causal:
            s = np.where(np.tril(np.ones((Nq, Nk), bool)), s, -np.inf)
        ref_lse = np.log(np.exp(s - s.max(1, keepdims=True)).sum(1)) + s.max(1)
        assert np.abs(lse - ref_lse).max() < 1e-12


def pin_descale_invariants(m):
    q8, k8, v8, (dq, dk, dv) = _inputs(3, 12, 20, 16)
    o, lse = m.attend_head_fp8(q8, k8, v8, dq, dk, dv, 0.2)
    # the value descale scales O linearly; it does not touch the weights
    o2, lse2 = m.attend_head_fp8(q8, k8, v8, dq, dk, 3.0 * dv, 0.2)
    assert np.allclose(o2, 3.0 * o, rtol=1e-13, atol=1e-15) and np.allclose(lse2, lse, rtol=0, atol=1e-13)
    # the q and k descales act like the softmax scale
    o3, lse3 = m.attend_head_fp8(q8, k8, v8, 2.0 * dq, dk, dv, 0.1)
    o4, lse4 = m.attend_head_fp8(q8, k8, v8, dq, 2.0 * dk, dv, 0.1)
    assert np.allclose(o3, o, rtol=1e-12, atol=1e-14) and np.allclose(o4, o, rtol=1e-12, atol=1e-14)
    assert np.allclose(lse3, lse, atol=1e-12) and np.allclose(lse4, lse, atol=1e-12)


def pin_quantizer_roundtrip(m):
    # the generator's codes reproduce its fp32 draws within e4m3 rounding:
    # relative 2^-4 for normal values, absolute 2^-10 * descale below 2^-6
    g = torch.Generator().manual_seed(11)
    x = torch.randn(1, 1, 64, 32, generator=g)
    (q8, _, _), (dq, _, _) = W.make_qkv_fp8(1, 1, 64, 32, 32, seed=11)
    back = m.dequantize(q8.numpy(), dq)
    xs = x.numpy().astype(np.float64)
    err = np.abs(back - xs)
    bound = np.maximum(2.0 ** -4 * np.abs(xs), 2.0 ** -10 * dq) + 1e-12
    assert np.all(err <= bound)
    assert abs(np.abs(back).max() - 448.0 * dq) < 1e-12 * dq    # amax maps to the largest code


PINS = [pin_decode_library, pin_decode_format_values, pin_attention_library, pin_descale_invariants,
        pin_quantizer_roundtrip]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(FP8)


MUTANTS = [
    ("exponent bias 8", "E4M3_BIAS = 7", "E4M3_BIAS = 8"),
    ("subnormals decoded as normals", "val = sign * np.where(e == 0, sub, normal)", "val = sign * normal"),
    ("sign dropped", "sign = np.where((c >> 7) & 1, -1.0, 1.0)", "sign = 1.0"),
    ("mantissa over 16", "normal = (1.0 + m / 8.0)", "normal = (1.0 + m / 16.0)"),
    ("k descale on v", "dequantize(v8, descale_v)", "dequantize(v8, descale_k)"),
    ("q descale dropped", "dequantize(q8, descale_q)", "dequantize(q8, 1.0)"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    src = inspect.getsource(FP8)
    assert src.count(old) == 1, f"mutation anchor not found: {old}"
    mod = types.ModuleType("oracle_fp8_mutant")
    exec(compile(src.replace(old, new), "oracle_fp8_mutant", "exec"), mod.__dict__)
    caught = 0
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, FloatingPointError):
            caught += 1
    assert caught > 0, f"no pin catches the mutant: {name}"
