"""Paged-KV decode attention for GB300 (sm_103a).

The compute lives in ``libpagedattn.so`` (hand-written CUDA, C ABI declared in
``include/pa.h``).  ``paged_kv_decode_cache_gb300.pa`` is the thin ctypes
binding with the same entry-point names; it loads the library on first use
and raises if it is missing.  ``workloads`` builds seeded synthetic inputs.
"""
from . import workloads  # noqa: F401  (inputs only; imports no CUDA code)

__all__ = ["workloads"]
