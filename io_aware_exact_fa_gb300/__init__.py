"""GB300-native exact attention forward pass (fused prefill + split-KV decode).

The compute path is the C-ABI library ``libfa_gb300.so`` (hand-written CUDA
for sm_103a). ``io_aware_exact_fa_gb300.fa`` is the thin Python binding over
it; importing that module raises if the library has not been built.
``io_aware_exact_fa_gb300.workloads`` draws seeded synthetic inputs.
"""

__all__ = ["fa", "workloads"]
