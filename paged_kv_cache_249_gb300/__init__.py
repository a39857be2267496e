"""Paged KV-cache decode attention for GB300 (sm_103a).

The CUDA library (libpagedkv.so, C ABI in include/pagedkv.h) holds the
kernels; ``pagedkv`` is its ctypes binding and ``workload`` the seeded
synthetic inputs.
"""
from . import workload  # noqa: F401

__all__ = ["workload", "pagedkv", "build"]
