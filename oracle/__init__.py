"""fp64 CPU oracle for exact attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this package:
only the tests, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline
leg and its ``--impl reference`` arm) may import or call it. It shares no code
with the CUDA path (no kernels, headers, helpers, tables or constants); both
sides only consume the same seeded input bytes.

Every function restates what the pages compute, in fp64, with NumPy:

* ``naive_attention`` -- the plain definition (scores, mask, softmax, weighted
  sum) that the fused kernel must reproduce up to rounding.
* ``online_attention`` -- the tile-by-tile online recurrence in the new-max
  form (running max m, running sum l, unnormalised output o, one rescale
  factor alpha per tile), generalised to d-dimensional values.
* ``online_row`` / ``blocklocal_row`` -- the same recurrence for one query
  row, in the new-max form and in the block-local-max form, used to pin the
  pages' worked examples with their intermediate states.
* ``merge_partials`` / ``splitkv_attention`` -- the two-block merge identity
  applied to per-split (m, l, o) triples, the arithmetic of split-KV decode.
* ``attention_grad.attend_head_grad`` / ``attention_grad.attention_grad`` --
  the backward pass: gradients of a loss through O with respect to Q, K and V
  (the chain rule through the definition, with the exact P).

* ``fp8.attend_head_fp8`` -- exact attention on e4m3 inputs: the 8-bit codes
  decoded field by field (``fp8.e4m3_decode``), times their descale factors,
  fed to the fp64 definition (pinned in tests/test_oracle_fp8.py).

Pins (tests/test_oracle.py): the pages' worked examples (tests/golden/),
agreement with torch's fp64 ``scaled_dot_product_attention`` and with
``scipy.special.logsumexp``, closed forms (one key, uniform scores, two keys),
shift invariance, key-permutation invariance, linearity in V, and brute force
over every mask of tiny rows.
"""

from .attention import (  # noqa: F401
    NEG_INF,
    allowed_mask,
    attend_head,
    naive_attention,
    online_attention,
    online_attention_head,
    online_row,
    blocklocal_row,
    merge_partials,
    splitkv_attention,
)
