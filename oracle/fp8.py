"""fp64 CPU oracle for the FP8 forward pass -- TEST INFRASTRUCTURE ONLY.

Only tests, ``__graft_entry__.smoke()`` and ``bench.py`` may import this
module; it imports nothing from the CUDA path.

Source: "FlashAttention: Attention Is Limited by Memory, Not Math", section
"FlashAttention 1, 2 and 3", which lists FP8 support among FlashAttention-3's
changes and says nothing more about it. The pages fix no FP8 arithmetic, so
this module takes the plainest reading (each point is also listed with the
design notes of the repository):

* The inputs are q, k and v as 8-bit e4m3 codes (1 sign bit, 4 exponent bits
  with bias 7, 3 mantissa bits; exponent field 0 holds the subnormals
  m * 2^-9; the codes with every exponent and mantissa bit set are NaN; there
  is no infinity), each tensor with one fp32 descale factor: the real value
  of a code c of q is decode(c) * descale_q, and likewise for k and v.
* What is computed is exact attention (the definition in ``attention.py``)
  on those real values: s_ij = scale * <q_i, k_j>, softmax over the visible
  keys, O = P V, lse = max + ln(sum). An implementation may round P to e4m3
  before the P V product; that rounding is an error of the implementation,
  bounded by the tolerance the tests state, not part of the definition.
"""

from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np

from oracle import attention as A

E4M3_BIAS = 7
E4M3_MAX = 448.0   # 0x7E: exponent field 15, mantissa 6 -> 2^8 * (1 + 6/8)


def e4m3_decode(codes) -> np.ndarray:
    """fp64 values of e4m3 codes (any integer array of bytes 0..255).

    Field by field: sign s = bit 7, exponent field e = bits 3..6, mantissa
    field m = bits 0..2. e = 0: (-1)^s * m / 8 * 2^(1 - bias) (zero and
    subnormals); e in 1..15: (-1)^s * (1 + m / 8) * 2^(e - bias), except that
    e = 15 with m = 7 is NaN (the format has no infinities)."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - E4M3_BIAS)
    sub = (m / 8.0) * 2.0 ** (1 - E4M3_BIAS)
    val = sign * np.where(e == 0, sub, normal)
    return np.where((e == 15) & (m == 7), np.nan, val)


def dequantize(codes, descale: float) -> np.ndarray:
    """Real values of an e4m3 tensor: decode(codes) * descale (fp64)."""
    return e4m3_decode(codes) * float(descale)


def attend_head_fp8(q8, k8, v8, descale_q: float, descale_k: float, descale_v: float, scale: float,
                    causal: bool = False, keep=None,
                    rows: Optional[Sequence[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Exact attention of one (batch, head) on e4m3 inputs: the codes are
    widened to fp64, multiplied by their descale factors, and passed to the
    fp64 definition ``attention.attend_head`` (q8 [Nq, d], k8 [Nk, d],
    v8 [Nk, dv] as byte arrays). Returns (O, lse) in fp64."""
    return A.attend_head(dequantize(q8, descale_q), dequantize(k8, descale_k), dequantize(v8, descale_v),
                         scale, causal, keep, rows=rows)
