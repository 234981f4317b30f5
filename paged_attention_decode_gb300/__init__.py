"""paged_attention_decode_gb300 -- fused paged-attention decode v2 for GB300 (sm_103a).

The compute path is ``libpa_v2.so`` (hand-written CUDA for sm_103a behind a C
ABI declared in ``include/pa_v2.h``); ``paged_attention_decode_gb300.pa_v2``
is its thin ctypes binding with the same names.  ``workloads`` builds seeded
synthetic inputs.  Importing this package loads nothing; the library is
loaded on the first call into the binding and raises if it is missing.
"""
__all__ = ["pa_v2", "workloads"]
