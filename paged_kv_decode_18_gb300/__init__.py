"""GB300-native (sm_103a) attention over a paged KV cache.

The CUDA library (``libpagedattn.so``, C ABI declared in ``include/pa.h``)
holds every step of the path; ``paged_kv_decode_18_gb300.binding`` is the thin
ctypes layer above it. Importing this package does not load the library: the
binding loads it on first use and raises if it is missing.
"""
__all__ = ["binding", "workloads"]
