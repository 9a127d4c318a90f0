"""GB300-native paged KV-cache attention: kv_append, paged decode attention
and chunked prefill attention, as hand-written sm_103a CUDA kernels behind a
C ABI (``include/pagedkv.h``).

Importing the package loads nothing; ``paged_kv_cache_104_gb300.binding``
loads the CUDA library on first use and raises if it is missing.
"""
__all__ = ["binding", "workloads", "build"]
