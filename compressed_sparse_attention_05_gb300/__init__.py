"""CSA2 compressed-sparse-attention layer step for one GB300 (sm_103a).

The compute path is libcsa2.so (hand-written CUDA behind the C ABI of
include/csa2.h); ``abi`` is its thin ctypes binding and ``harness`` lays a
workload out in device memory.  Build with ``python -m
compressed_sparse_attention_05_gb300.build``.  There is no CPU fallback: the
entry points raise if the library is missing.
"""
from . import abi  # noqa: F401

__all__ = ["abi", "harness", "build"]
