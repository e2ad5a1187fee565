"""GB300-native DSA decode hot path (index scores -> top-k -> FP8 gather-attend).

The compute lives in ``libdsa_gb300.so`` (hand-written CUDA for sm_103a behind
a C ABI declared in ``include/dsa.h``).  ``sparse_attention_mla_dsa_gb300.api``
is a thin ctypes binding with the same entry-point names; importing this
package does not load the library, so CPU-only tooling (the input generator)
works without a GPU.
"""
__all__ = ["api", "workloads"]
