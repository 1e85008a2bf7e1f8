"""Thin Python binding over the kv4 C ABI (include/kv4.h).

Argument marshalling only: every step of the path runs in the CUDA kernels of
libkv4.so.  PyTorch tensors supply device memory and the current CUDA stream.
Functions keep the C names.  If the library is missing this module raises --
there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkv4.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "kv4.h")

KV4_OK = 0
KV4_ERR_INVALID_ARG = 1
KV4_ERR_UNSUPPORTED = 2
KV4_ERR_LAUNCH = 3
KV4_ERR_WORKSPACE = 4

KV4_STATUS_BAD_PAGE = 1
KV4_STATUS_BAD_POS = 2
KV4_STATUS_BAD_SEQ = 4
KV4_STATUS_NONFINITE = 8
KV4_STATUS_BAD_LEN = 16
KV4_STATUS_TIMEOUT = 32
KV4_STATUS_INTERNAL = 64
KV4_STATUS_V_RANGE = 128

KV4_KERNEL_AUTO = 0
KV4_KERNEL_CUDA_CORE = 1
KV4_KERNEL_MMA_SYNC = 2
KV4_KERNEL_STREAM = 4


class kv4_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_q_heads", "num_kv_heads", "head_dim", "page_size", "int4_group", "int8_group",
        "sink", "recent", "max_seqs", "num_pages", "max_pages_per_seq")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


def make_layout(*, h_q=32, h_kv=8, d_h=128, group=32, sink=4, recent=128, max_seqs,
                num_pages, max_pages_per_seq) -> kv4_layout:
    return kv4_layout(h_q, h_kv, d_h, 16, group, d_h, sink, recent, max_seqs, num_pages,
                      max_pages_per_seq)


class KV4Error(RuntimeError):
    pass


_lib = None


def declared_symbols():
    """Function names declared in include/kv4.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(kv4_[a-z0-9_]+)\s*\(", text)))


def load(build_if_missing: bool = False):
    """Load libkv4.so (optionally building it first).  Raises if unavailable."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        if build_if_missing:
            from . import build as _b
            _b.build()
        else:
            raise KV4Error(f"{LIB_PATH} is missing: build it with "
                           "`python -m int8_kv_cache_kv4_gb300.build` (no CPU fallback exists)")
    try:
        import torch  # noqa: F401  (loads the shared CUDA runtime first)
    except Exception:
        pass
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    I = ctypes.c_int32
    Sz = ctypes.c_size_t
    LP = ctypes.POINTER(kv4_layout)
    sig = {
        "kv4_abi_version": (ctypes.c_int, []),
        "kv4_set_decode_kernel": (ctypes.c_int, [ctypes.c_int]),
        "kv4_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "kv4_check_layout": (ctypes.c_int, [LP]),
        "kv4_paged_cache_bytes": (Sz, [LP]),
        "kv4_side_cache_bytes": (Sz, [LP]),
        "kv4_bf16_cache_bytes": (Sz, [LP]),
        "kv4_num_splits": (I, [LP, I, I]),
        "kv4_workspace_bytes": (Sz, [LP, I, I]),
        "kv4_bf16_workspace_bytes": (Sz, [LP, I, I]),
        "kv4_quant_append": (ctypes.c_int, [LP, P, P, P, P, P, P, I, P, P, P, P]),
        "kv4_quant_append_hadamard": (ctypes.c_int, [LP, P, P, P, P, P, P, I, P, P, P, P]),
        "kv4_hadamard_bf16": (ctypes.c_int, [P, P, I, I, P]),
        "kv4_fp4_cache_bytes": (Sz, [LP]),
        "kv4_fp4_append": (ctypes.c_int, [LP, I, I, P, P, P, P, P, I, P, P, P, P]),
        "kv4_fp4_to_bf16": (ctypes.c_int, [LP, I, P, P, P]),
        "kv4_decode_attn": (ctypes.c_int, [LP, P, P, P, P, I, P, ctypes.c_float, I, P, Sz, P, P,
                                           P, P]),
        "kv4_decode_attn_hadamard": (ctypes.c_int, [LP, P, P, P, P, I, P, ctypes.c_float, I, P, Sz, P, P,
                                           P, P]),
        "kv4_split_combine": (ctypes.c_int, [P, P, I, I, I, P, P, P]),
        "kv4_bf16_append": (ctypes.c_int, [LP, P, P, P, P, P, I, P, P, P, P]),
        "kv4_bf16_decode_attn": (ctypes.c_int, [LP, P, P, P, I, P, ctypes.c_float, I, P, Sz, P,
                                                P, P, P]),
        "kv4_noalloc_scratch_bytes": (Sz, []),
        "kv4_decode_attn_noalloc": (ctypes.c_int, [LP, P, P, P, P, I, P, ctypes.c_float, I, P, P,
                                                   P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


# ------------------------------------------------------------- marshalling

def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(rc: int, what: str):
    if rc != KV4_OK:
        msg = load().kv4_status_string(rc).decode()
        raise KV4Error(f"{what}: {msg} (code {rc})")


def _dev(t, dtype, name):
    import torch
    if t is None:
        return
    if not t.is_cuda:
        raise KV4Error(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise KV4Error(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise KV4Error(f"{name} must be contiguous")


def kv4_set_decode_kernel(which: int) -> int:
    """Select the decode kernel (KV4_KERNEL_*); returns the previous choice."""
    return int(load().kv4_set_decode_kernel(int(which)))


def paged_cache_bytes(layout: kv4_layout) -> int:
    return int(load().kv4_paged_cache_bytes(ctypes.byref(layout)))


def side_cache_bytes(layout: kv4_layout) -> int:
    return int(load().kv4_side_cache_bytes(ctypes.byref(layout)))


def bf16_cache_bytes(layout: kv4_layout) -> int:
    return int(load().kv4_bf16_cache_bytes(ctypes.byref(layout)))


def num_splits(layout: kv4_layout, num_seqs: int, max_splits: int = 0) -> int:
    return int(load().kv4_num_splits(ctypes.byref(layout), num_seqs, max_splits))


def workspace_bytes(layout: kv4_layout, num_seqs: int, max_splits: int = 0) -> int:
    return int(load().kv4_workspace_bytes(ctypes.byref(layout), num_seqs, max_splits))


def bf16_workspace_bytes(layout: kv4_layout, num_seqs: int, max_splits: int = 0) -> int:
    return int(load().kv4_bf16_workspace_bytes(ctypes.byref(layout), num_seqs, max_splits))


def kv4_quant_append(layout, paged, side, k_new, v_new, tok_seq, tok_pos, seq_lens, block_table,
                     status=None, stream=None):
    """Quantize-on-append of T tokens (k_new/v_new bf16 [T][h_kv][d_h])."""
    _quant_append("kv4_quant_append", layout, paged, side, k_new, v_new, tok_seq, tok_pos,
                  seq_lens, block_table, status, stream)


def kv4_quant_append_hadamard(layout, paged, side, k_new, v_new, tok_seq, tok_pos, seq_lens,
                              block_table, status=None, stream=None):
    """kv4_quant_append with K rotated by the normalized Hadamard matrix first."""
    _quant_append("kv4_quant_append_hadamard", layout, paged, side, k_new, v_new, tok_seq,
                  tok_pos, seq_lens, block_table, status, stream)


def kv4_hadamard_bf16(x, y=None, stream=None):
    """Rotate every row of x (bf16 [..., d], d = 64 or 128) by the normalized
    Hadamard matrix into y (default: in place).  Returns y."""
    import torch
    _dev(x, torch.bfloat16, "x")
    if y is None:
        y = x
    _dev(y, torch.bfloat16, "y")
    if y.shape != x.shape:
        raise KV4Error("kv4_hadamard_bf16: x and y differ in shape")
    d = int(x.shape[-1]) if x.dim() else 0
    rows = x.numel() // d if d else 0
    rc = load().kv4_hadamard_bf16(_ptr(x), _ptr(y), rows, d, _stream(stream))
    _check(rc, "kv4_hadamard_bf16")
    return y


KV4_FP4_NVFP4, KV4_FP4_MXFP4 = 1, 2


def fp4_cache_bytes(layout: kv4_layout) -> int:
    return int(load().kv4_fp4_cache_bytes(ctypes.byref(layout)))


def kv4_fp4_append(layout, fmt, cache, k_new, v_new, tok_seq, tok_pos, seq_lens, block_table,
                   rotate_k=False, status=None, stream=None):
    """FP4 probe append (NVFP4 or MXFP4) of T tokens, k_new/v_new bf16 [T][h_kv][d_h]."""
    import torch
    _dev(cache, torch.uint8, "cache")
    for n, t in (("k_new", k_new), ("v_new", v_new)):
        _dev(t, torch.bfloat16, n)
    for n, t in (("tok_seq", tok_seq), ("tok_pos", tok_pos), ("seq_lens", seq_lens),
                 ("block_table", block_table), ("status", status)):
        _dev(t, torch.int32, n)
    T = int(tok_seq.numel())
    if tok_pos.numel() != T or k_new.numel() != T * layout.num_kv_heads * layout.head_dim:
        raise KV4Error("kv4_fp4_append: token arrays disagree in length")
    _check(load().kv4_fp4_append(ctypes.byref(layout), int(fmt), 1 if rotate_k else 0, _ptr(cache),
                                 _ptr(k_new), _ptr(v_new), _ptr(tok_seq), _ptr(tok_pos), T,
                                 _ptr(seq_lens), _ptr(block_table), _ptr(status), _stream(stream)),
           "kv4_fp4_append")


def kv4_fp4_to_bf16(layout, fmt, cache, bf16_cache, stream=None):
    """Reconstruct the whole FP4 probe pool into the bf16 comparator layout."""
    import torch
    _dev(cache, torch.uint8, "cache")
    _dev(bf16_cache, torch.uint8, "bf16_cache")
    _check(load().kv4_fp4_to_bf16(ctypes.byref(layout), int(fmt), _ptr(cache), _ptr(bf16_cache),
                                  _stream(stream)), "kv4_fp4_to_bf16")


def _quant_append(name, layout, paged, side, k_new, v_new, tok_seq, tok_pos, seq_lens,
                  block_table, status, stream):
    import torch
    _dev(paged, torch.uint8, "paged")
    _dev(side, torch.uint8, "side")
    for n, t in (("k_new", k_new), ("v_new", v_new)):
        _dev(t, torch.bfloat16, n)
    for n, t in (("tok_seq", tok_seq), ("tok_pos", tok_pos), ("seq_lens", seq_lens),
                 ("block_table", block_table), ("status", status)):
        _dev(t, torch.int32, n)
    T = int(tok_seq.numel())
    if tok_pos.numel() != T or k_new.numel() != T * layout.num_kv_heads * layout.head_dim:
        raise KV4Error(f"{name}: token arrays disagree in length")
    rc = getattr(load(), name)(ctypes.byref(layout), _ptr(paged), _ptr(side), _ptr(k_new),
                               _ptr(v_new), _ptr(tok_seq), _ptr(tok_pos), T, _ptr(seq_lens),
                               _ptr(block_table), _ptr(status), _stream(stream))
    _check(rc, name)


def _check_decode_args(name, layout, paged, side, q, seq_lens, block_table, out, out_lse, status):
    """Types, devices and shapes of a decode call's tensors, so that a
    mis-sized tensor is a KV4Error here instead of an out-of-bounds access on
    the device.  Returns the number of sequences B = q.shape[0]."""
    import torch
    _dev(paged, torch.uint8, "paged")
    _dev(side, torch.uint8, "side")
    _dev(q, torch.bfloat16, "q")
    _dev(out, torch.bfloat16, "out")
    _dev(out_lse, torch.float32, "out_lse")
    _dev(seq_lens, torch.int32, "seq_lens")
    _dev(block_table, torch.int32, "block_table")
    _dev(status, torch.int32, "status")
    shape = (layout.num_q_heads, layout.head_dim)
    if q.dim() != 3 or tuple(q.shape[1:]) != shape or not q.is_contiguous():
        raise KV4Error(f"{name}: q must be a contiguous [B][{shape[0]}][{shape[1]}] tensor")
    B = int(q.shape[0])
    if tuple(out.shape) != tuple(q.shape) or not out.is_contiguous():
        raise KV4Error(f"{name}: out must be contiguous and shaped like q")
    if out_lse is not None and (tuple(out_lse.shape) != (B, layout.num_q_heads)
                                or not out_lse.is_contiguous()):
        raise KV4Error(f"{name}: out_lse must be a contiguous [B][h_q] tensor")
    if seq_lens.numel() < B or B > layout.max_seqs:
        raise KV4Error(f"{name}: seq_lens holds fewer than B entries or B > max_seqs")
    if tuple(block_table.shape) != (layout.max_seqs, layout.max_pages_per_seq) or \
            not block_table.is_contiguous():
        raise KV4Error(f"{name}: block_table must be a contiguous [max_seqs][max_pages_per_seq] tensor")
    if paged.numel() < paged_cache_bytes(layout) or \
            (layout.sink + layout.recent > 0 and side.numel() < side_cache_bytes(layout)):
        raise KV4Error(f"{name}: cache buffers smaller than the layout's sizes")
    if status is not None and status.numel() < 1:
        raise KV4Error(f"{name}: status must hold one int32")
    return B


def kv4_decode_attn(layout, paged, side, q, seq_lens, block_table, workspace, out, out_lse=None,
                    sm_scale=None, max_splits=0, status=None, stream=None, rotate_q=False):
    """Split-KV GQA decode attention; q/out bf16 [B][h_q][d_h].  rotate_q:
    kv4_decode_attn_hadamard (the query rotated by the call, for a cache
    written with the Hadamard K-rotation)."""
    import torch
    name = "kv4_decode_attn_hadamard" if rotate_q else "kv4_decode_attn"
    B = _check_decode_args(name, layout, paged, side, q, seq_lens, block_table, out, out_lse,
                           status)
    _dev(workspace, torch.uint8, "workspace")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(layout.head_dim)
    rc = getattr(load(), name)(ctypes.byref(layout), _ptr(paged), _ptr(side), _ptr(q),
                               _ptr(seq_lens), B, _ptr(block_table), float(sm_scale),
                               int(max_splits), _ptr(workspace), workspace.numel(), _ptr(out),
                               _ptr(out_lse), _ptr(status), _stream(stream))
    _check(rc, name)


def kv4_split_combine(part_o, part_lse, out, out_lse=None, stream=None):
    """Eq. A1 merge: part_o fp32 [rows][n][d], part_lse fp32 [rows][n] -> out bf16 [rows][d]."""
    import torch
    _dev(part_o, torch.float32, "part_o")
    _dev(part_lse, torch.float32, "part_lse")
    _dev(out, torch.bfloat16, "out")
    _dev(out_lse, torch.float32, "out_lse")
    rows, n, d = part_o.shape
    rc = load().kv4_split_combine(_ptr(part_o), _ptr(part_lse), rows, n, d, _ptr(out),
                                  _ptr(out_lse), _stream(stream))
    _check(rc, "kv4_split_combine")


def kv4_bf16_append(layout, cache, k_new, v_new, tok_seq, tok_pos, seq_lens, block_table,
                    status=None, stream=None):
    import torch
    _dev(cache, torch.uint8, "cache")
    T = int(tok_seq.numel())
    rc = load().kv4_bf16_append(ctypes.byref(layout), _ptr(cache), _ptr(k_new), _ptr(v_new),
                                _ptr(tok_seq), _ptr(tok_pos), T, _ptr(seq_lens),
                                _ptr(block_table), _ptr(status), _stream(stream))
    _check(rc, "kv4_bf16_append")


def kv4_bf16_decode_attn(layout, cache, q, seq_lens, block_table, workspace, out, out_lse=None,
                         sm_scale=None, max_splits=0, status=None, stream=None):
    import torch
    _dev(cache, torch.uint8, "cache")
    _dev(q, torch.bfloat16, "q")
    _dev(out, torch.bfloat16, "out")
    B = int(q.shape[0])
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(layout.head_dim)
    rc = load().kv4_bf16_decode_attn(ctypes.byref(layout), _ptr(cache), _ptr(q), _ptr(seq_lens),
                                     B, _ptr(block_table), float(sm_scale), int(max_splits),
                                     _ptr(workspace), workspace.numel(), _ptr(out), _ptr(out_lse),
                                     _ptr(status), _stream(stream))
    _check(rc, "kv4_bf16_decode_attn")


def kv4_decode_attn_noalloc(layout, paged, side, q, seq_lens, block_table, out, out_lse=None,
                            sm_scale=None, max_splits=0, status=None, stream=None):
    """kv4_decode_attn without a caller workspace, for callers that cannot
    allocate device memory: the library's fixed scratch array is used instead
    (see include/kv4.h for its size, first-call set-up and sharing rules)."""
    B = _check_decode_args("kv4_decode_attn_noalloc", layout, paged, side, q, seq_lens,
                           block_table, out, out_lse, status)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(layout.head_dim)
    rc = load().kv4_decode_attn_noalloc(ctypes.byref(layout), _ptr(paged), _ptr(side), _ptr(q),
                                        _ptr(seq_lens), B, _ptr(block_table), float(sm_scale),
                                        int(max_splits), _ptr(out), _ptr(out_lse), _ptr(status),
                                        _stream(stream))
    _check(rc, "kv4_decode_attn_noalloc")
