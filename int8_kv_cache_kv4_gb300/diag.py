"""Binding of the tensor-pipe rate probe (include/kv4_diag.h, libkv4_diag.so).

Not part of the decode library: only the benchmark's report mode loads it.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkv4_diag.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "kv4_diag.h")

# kinds: warp-level fp16 and int8 MMA, tcgen05 kind::f16 (128 x 256 x 16)
KIND_MMA_F16, KIND_MMA_I8, KIND_TC_F16 = 0, 1, 2
OPS_PER_MMA = {KIND_MMA_F16: 4096, KIND_MMA_I8: 8192, KIND_TC_F16: 2 * 128 * 256 * 16}
THREADS = {KIND_MMA_F16: 256, KIND_MMA_I8: 256, KIND_TC_F16: 128}
ISSUERS_PER_CTA = {KIND_MMA_F16: 8 * 4, KIND_MMA_I8: 8 * 4, KIND_TC_F16: 1}

_lib = None


def declared_symbols():
    return sorted(set(re.findall(r"\b(kv4_[a-z0-9_]+)\s*\(", open(HEADER).read())))


def load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m int8_kv_cache_kv4_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        lib.kv4_diag_mma_rate.restype = ctypes.c_int
        lib.kv4_diag_mma_rate.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_void_p, ctypes.c_void_p]
        _lib = lib
    return _lib


def kv4_diag_mma_rate(kind, blocks, iters, sink, stream=None):
    """Launch the probe on the current (or given) stream; sink: int32 device tensor."""
    import torch
    st = (stream or torch.cuda.current_stream()).cuda_stream
    rc = load().kv4_diag_mma_rate(int(kind), int(blocks), int(iters),
                                  ctypes.c_void_p(sink.data_ptr()), ctypes.c_void_p(st))
    if rc != 0:
        raise RuntimeError(f"kv4_diag_mma_rate failed with code {rc}")


def ops(kind, blocks, iters):
    """Multiply-adds x 2 performed by one launch."""
    return blocks * ISSUERS_PER_CTA[kind] * iters * OPS_PER_MMA[kind]
