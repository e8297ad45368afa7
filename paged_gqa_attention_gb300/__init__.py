"""GB300-native paged grouped-query attention.

The compute lives in ``libpagedattn.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/pagedattn.h``).  This package holds the thin ctypes binding
(``ops``), the build step (``build``) and the seeded workload generators
(``workloads``).  Importing the package does not load the library; the first call
into ``ops`` does, and fails loudly if the library is missing.
"""
__all__ = ["ops", "workloads", "build"]
