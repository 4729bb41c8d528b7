"""Paged KV-cache decode attention for one GB300 GPU.

The hot path lives in the CUDA library ``_lib/libpa.so`` (C ABI in
``include/pa.h``); ``paged_kv_cache_251_gb300.pa`` is its thin binding, and
``paged_kv_cache_251_gb300.blocks`` the host-side block manager.  Importing
this package loads neither, so the input generators in ``workloads`` work on
machines without a GPU.
"""
__version__ = "0.1.0"
