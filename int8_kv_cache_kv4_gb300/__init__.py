"""GB300-native KV4-RL decode hot path: mixed INT4/INT8 paged KV cache.

The compute path is libkv4.so (hand-written sm_103a CUDA kernels behind the C
ABI in include/kv4.h); ``kv4`` is its thin ctypes binding and ``workloads``
holds the seeded synthetic inputs.
"""
from . import kv4, workloads  # noqa: F401
