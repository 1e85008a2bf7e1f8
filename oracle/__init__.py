"""CPU oracle for the KV4-RL mixed INT4/INT8 KV cache (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It is never on the product path and shares no code
with the CUDA library: the C source ``kv4_oracle.c`` restates the paper's steps
(KV4-RL, Sec. 3 eq. 3.3, Sec. 5.1-5.3, App. A.3 eq. A1) in plain C with
explicit IEEE-754 rounding, and this module is only a ctypes wrapper over it
plus numpy marshalling.

Every function here is pinned in ``tests/test_oracle_*.py`` against closed
forms, invariants, library routines and brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kv4_oracle.c")
_SRC_FP4 = os.path.join(_HERE, "kv4_fp4_oracle.c")
_LIB = os.path.join(_HERE, "libkv4_oracle.so")
_lock = threading.Lock()
_lib = None

RNE, DOWN, UP = 0, 1, 2
ST_BAD_PAGE, ST_BAD_POS, ST_BAD_SEQ, ST_NONFINITE = 1, 2, 4, 8

PAGE = 16


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction, dynamic
    rounding modes honoured).  Returns the library path."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_SRC_FP4))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-std=c11", "-O1", "-frounding-math", "-fno-fast-math",
               "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC, _SRC_FP4, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            Lg = ctypes.c_long
            D = ctypes.c_double
            lib.kv4o_f32_to_f16.restype = ctypes.c_uint16
            lib.kv4o_f32_to_f16.argtypes = [ctypes.c_float, I]
            lib.kv4o_f16_to_f32.restype = ctypes.c_float
            lib.kv4o_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.kv4o_f32_to_f16_n.argtypes = [P, Lg, I, P]
            lib.kv4o_sub_dir_n.argtypes = [P, P, Lg, I, P]
            lib.kv4o_div_dir_n.argtypes = [P, P, Lg, I, P]
            lib.kv4o_int4_encode_n.argtypes = [P, Lg, I, P, P, P]
            lib.kv4o_int4_encode_n.restype = I
            lib.kv4o_int8_encode_n.argtypes = [P, Lg, I, P, P]
            lib.kv4o_int8_encode_n.restype = I
            lib.kv4o_is_protected.argtypes = [I, I, I, I]
            lib.kv4o_is_protected.restype = I
            lib.kv4o_side_slot.argtypes = [I, I, I]
            lib.kv4o_side_slot.restype = I
            lib.kv4o_quant_append.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, P, P, I, P, P, I]
            lib.kv4o_quant_append.restype = I
            lib.kv4o_dequant_seq.argtypes = [I, I, I, I, I, I, P, P, P, P, I]
            lib.kv4o_hadamard_f32_n.argtypes = [P, Lg, I]
            lib.kv4o_hadamard_f32_n.restype = None
            lib.fp4o_e2m1_round_n.argtypes = [P, Lg, P]
            lib.fp4o_e2m1_round_n.restype = None
            lib.fp4o_e4m3_round_n.argtypes = [P, Lg, P]
            lib.fp4o_e4m3_round_n.restype = None
            lib.fp4o_e2m1_value.argtypes = [I]
            lib.fp4o_e2m1_value.restype = ctypes.c_float
            lib.fp4o_e4m3_value.argtypes = [I]
            lib.fp4o_e4m3_value.restype = ctypes.c_float
            lib.fp4o_encode_n.argtypes = [I, P, Lg, I, P, P, P]
            lib.fp4o_encode_n.restype = I
            lib.fp4o_decode_n.argtypes = [I, P, P, P, Lg, I, P]
            lib.fp4o_decode_n.restype = None
            lib.fp4o_append.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, I, P, P]
            lib.fp4o_append.restype = I
            lib.fp4o_dequant_seq.argtypes = [I, I, I, I, I, P, P, P, P]
            lib.fp4o_dequant_seq.restype = I
            lib.kv4o_dequant_seq.restype = I
            lib.kv4o_attend.argtypes = [I, I, I, I, P, P, P, D, P, P, P]
            lib.kv4o_attend.restype = None
            lib.kv4o_combine.argtypes = [I, I, P, P, P, P]
            lib.kv4o_combine.restype = None
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ scalars

def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact widening)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    lib = _get()
    return np.array([lib.kv4o_f16_to_f32(int(v)) for v in h.ravel()], dtype=np.float32).reshape(h.shape)


def f32_to_f16(x: np.ndarray, mode: int) -> np.ndarray:
    """float32 -> fp16 bits with rounding ``mode`` (RNE, DOWN or UP)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _get().kv4o_f32_to_f16_n(_p(x), x.size, mode, _p(out))
    return out


def sub_dir(a: np.ndarray, b: np.ndarray, mode: int) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.float32)
    _get().kv4o_sub_dir_n(_p(a), _p(b), a.size, mode, _p(out))
    return out


def div_dir(a: np.ndarray, b: np.ndarray, mode: int) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.float32)
    _get().kv4o_div_dir_n(_p(a), _p(b), a.size, mode, _p(out))
    return out


# ----------------------------------------------------------------- encoders

def int4_encode(x: np.ndarray, g: int):
    """INT4 affine encode along the last axis in groups of ``g`` (KV4-RL eq. 3.3,
    Sec. 5.1).  x: float32 [..., n], n % g == 0.
    Returns (codes uint8 [..., n], delta16 uint16 [..., n/g], off16 uint16
    [..., n/g], status)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n = x.shape[-1]
    assert n % g == 0
    ng = x.size // g
    codes = np.empty(x.shape, dtype=np.uint8)
    d16 = np.empty(x.shape[:-1] + (n // g,), dtype=np.uint16)
    m16 = np.empty_like(d16)
    st = _get().kv4o_int4_encode_n(_p(x), ng, g, _p(codes), _p(d16), _p(m16))
    return codes, d16, m16, st


def int8_encode(x: np.ndarray):
    """INT8 symmetric encode of each vector along the last axis (KV4-RL App. A.3).
    Returns (codes int8, scale16 uint16 [...], status)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n = x.shape[-1]
    codes = np.empty(x.shape, dtype=np.int8)
    s16 = np.empty(x.shape[:-1], dtype=np.uint16)
    st = _get().kv4o_int8_encode_n(_p(x), x.size // n, n, _p(codes), _p(s16))
    return codes, s16, st


def is_protected(p: int, L: int, S: int, R: int) -> bool:
    return bool(_get().kv4o_is_protected(p, L, S, R))


def side_slot(p: int, S: int, R: int) -> int:
    return int(_get().kv4o_side_slot(p, S, R))


# ------------------------------------------------------------ packed layout

def chunk_bytes(d_h: int, g: int) -> int:
    return 16 * d_h + 128 * (d_h // g)


def side_scale_entries(S: int, R: int) -> int:
    """Entries of each side-cache scale array: S + R rounded up to 8."""
    return (S + R + 7) // 8 * 8


def side_block_bytes(d_h: int, S: int, R: int) -> int:
    return 2 * (S + R) * d_h + 4 * side_scale_entries(S, R)


def quant_append(*, h_kv, d_h, g, S, R, max_seqs, num_pages, max_pages_per_seq,
                 paged: np.ndarray, side: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
                 tok_seq: np.ndarray, tok_pos: np.ndarray, seq_lens: np.ndarray,
                 block_table: np.ndarray, rotate_k: bool = False) -> int:
    """Write T new tokens into the packed cache bytes ``paged`` / ``side`` in place.
    k_new/v_new: bf16 bits uint16 [T][h_kv][d_h].  rotate_k: K is rotated by
    hadamard_f32 before it is quantized (V never is).  Returns status bits."""
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    tok_seq = np.ascontiguousarray(tok_seq, dtype=np.int32)
    tok_pos = np.ascontiguousarray(tok_pos, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    assert paged.dtype == np.uint8 and side.dtype == np.uint8
    assert paged.size >= num_pages * h_kv * chunk_bytes(d_h, g)
    assert side.size >= max_seqs * h_kv * side_block_bytes(d_h, S, R)
    T = int(tok_seq.size)
    return int(_get().kv4o_quant_append(h_kv, d_h, g, S, R, max_seqs, num_pages,
                                        max_pages_per_seq, _p(paged), _p(side), _p(k_new),
                                        _p(v_new), _p(tok_seq), _p(tok_pos), T, _p(seq_lens),
                                        _p(block_table), 1 if rotate_k else 0))


# ----------------------------------------------------------------- decoding

def dequant_seq(k_src: np.ndarray, v_src: np.ndarray, *, g: int, S: int, R: int,
                rotate_k: bool = False):
    """Dequantized cache of one sequence (fp64).  k_src/v_src: bf16 bits
    [h_kv][L][d_h].  Protected positions decode INT8, the rest INT4.
    rotate_k: K is rotated (hadamard_f32) before it is quantized."""
    k_src = np.ascontiguousarray(k_src, dtype=np.uint16)
    v_src = np.ascontiguousarray(v_src, dtype=np.uint16)
    h_kv, L, d_h = k_src.shape
    kh = np.empty((h_kv, L, d_h), dtype=np.float64)
    vh = np.empty_like(kh)
    st = _get().kv4o_dequant_seq(h_kv, d_h, g, S, R, L, _p(k_src), _p(v_src), _p(kh), _p(vh),
                                 1 if rotate_k else 0)
    return kh, vh, st


def attend(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, sm_scale: float):
    """fp64 softmax attention of one sequence.  q: bf16 bits [h_q][d_h];
    k_hat/v_hat: float64 [h_kv][L][d_h].  Returns (out [h_q][d_h], lse [h_q])."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_hat = np.ascontiguousarray(k_hat, dtype=np.float64)
    v_hat = np.ascontiguousarray(v_hat, dtype=np.float64)
    h_q, d_h = q.shape
    h_kv, L, _ = k_hat.shape
    out = np.empty((h_q, d_h), dtype=np.float64)
    lse = np.empty((h_q,), dtype=np.float64)
    scratch = np.empty((max(L, 1),), dtype=np.float64)
    _get().kv4o_attend(h_q, h_kv, d_h, L, _p(q), _p(k_hat), _p(v_hat), float(sm_scale),
                       _p(out), _p(lse), _p(scratch))
    return out, lse


def decode_seq(q: np.ndarray, k_src: np.ndarray, v_src: np.ndarray, *, g: int, S: int, R: int,
               sm_scale: float, rotate_k: bool = False):
    """Quantize one sequence's source K/V with the protection rule, then attend.
    rotate_k: K is rotated before quantization (q must then be the rotated
    query).  Returns (out fp64 [h_q][d_h], lse fp64 [h_q], status)."""
    kh, vh, st = dequant_seq(k_src, v_src, g=g, S=S, R=R, rotate_k=rotate_k)
    out, lse = attend(q, kh, vh, sm_scale)
    return out, lse, st


def combine(o_parts: np.ndarray, z_parts: np.ndarray):
    """Eq. A1 merge of n partial results.  o_parts [n][d], z_parts [n]."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    z_parts = np.ascontiguousarray(z_parts, dtype=np.float64)
    n, d = o_parts.shape
    out = np.empty((d,), dtype=np.float64)
    z = np.empty((1,), dtype=np.float64)
    _get().kv4o_combine(n, d, _p(o_parts), _p(z_parts), _p(out), _p(z))
    return out, float(z[0])


def hadamard_f32(x: np.ndarray) -> np.ndarray:
    """Normalized Sylvester-Hadamard rotation of every row of x (float32, last
    axis a power of two) in fp32, in the fixed order kv4o_hadamard_f32 states."""
    x = np.array(x, dtype=np.float32, order="C", copy=True)
    n = x.shape[-1]
    assert n > 0 and n & (n - 1) == 0
    _get().kv4o_hadamard_f32_n(_p(x), x.size // n, n)
    return x


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def hadamard_bf16(bits: np.ndarray) -> np.ndarray:
    """Rotated query rows: bf16 bits in, hadamard_f32 of their values, rounded
    to bf16 (nearest even) bits out."""
    return f32_to_bf16_bits(hadamard_f32(bf16_to_f32(np.asarray(bits, dtype=np.uint16))))


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp64/fp32 -> nearest-even bf16, returned as float64 (for output checks)."""
    f = np.ascontiguousarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint32) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


# ------------------------------------------------------------ FP4 probe formats
# (kv4_fp4_oracle.c: NVFP4 and MXFP4 as KV4-RL App. D.4 compares them)

NVFP4, MXFP4 = 1, 2


def e2m1_round(y: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code (uint8, sign in bit 3) of every fp32 value."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty(y.shape, dtype=np.uint8)
    _get().fp4o_e2m1_round_n(_p(y), y.size, _p(out))
    return out


def e2m1_value(code: int) -> float:
    return float(_get().fp4o_e2m1_value(int(code)))


def e4m3_round(t: np.ndarray) -> np.ndarray:
    t = np.ascontiguousarray(t, dtype=np.float32)
    out = np.empty(t.shape, dtype=np.uint8)
    _get().fp4o_e4m3_round_n(_p(t), t.size, _p(out))
    return out


def e4m3_value(code: int) -> float:
    return float(_get().fp4o_e4m3_value(int(code)))


def fp4_encode(x: np.ndarray, fmt: int):
    """Encode every row (last axis n) of x (fp32): codes uint8 [.., n] (one
    E2M1 code per element), block scales uint8 [.., n/16 | n/32], global
    scales fp32 [..] (NVFP4; zero for MXFP4), status."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n = x.shape[-1]
    nv = x.size // n
    nb = n // 16 if fmt == NVFP4 else n // 32
    codes = np.empty(x.shape, dtype=np.uint8)
    bs = np.empty(x.shape[:-1] + (nb,), dtype=np.uint8)
    g = np.zeros(x.shape[:-1], dtype=np.float32)
    st = _get().fp4o_encode_n(fmt, _p(x), nv, n, _p(codes), _p(bs), _p(g))
    return codes, bs, g, st


def fp4_decode(codes: np.ndarray, bs: np.ndarray, g: np.ndarray, fmt: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    bs = np.ascontiguousarray(bs, dtype=np.uint8)
    g = np.ascontiguousarray(g, dtype=np.float32)
    n = codes.shape[-1]
    out = np.empty(codes.shape, dtype=np.float32)
    _get().fp4o_decode_n(fmt, _p(codes), _p(bs), _p(g), codes.size // n, n, _p(out))
    return out


def fp4_row_bytes(d_h: int) -> int:
    return d_h // 2 + 16


def fp4_append(*, h_kv, d_h, fmt, rotate_k=False, max_seqs, num_pages, max_pages_per_seq,
               cache: np.ndarray, k_new, v_new, tok_seq, tok_pos, seq_lens, block_table) -> int:
    """Write T tokens into the packed FP4 probe cache bytes in place."""
    T = int(len(tok_seq))
    if T == 0:
        return 0
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    tok_seq = np.ascontiguousarray(tok_seq, dtype=np.int32)
    tok_pos = np.ascontiguousarray(tok_pos, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    return int(_get().fp4o_append(h_kv, d_h, fmt, 1 if rotate_k else 0, max_seqs, num_pages,
                                  max_pages_per_seq, _p(cache), _p(k_new), _p(v_new),
                                  _p(tok_seq), _p(tok_pos), T, _p(seq_lens), _p(block_table)))


def fp4_dequant_seq(k_src: np.ndarray, v_src: np.ndarray, *, fmt: int, rotate_k: bool = False):
    """The probe's bf16 attention operands of one sequence (fp64 [h_kv][L][d_h])."""
    k_src = np.ascontiguousarray(k_src, dtype=np.uint16)
    v_src = np.ascontiguousarray(v_src, dtype=np.uint16)
    h_kv, L, d_h = k_src.shape
    kh = np.empty((h_kv, L, d_h))
    vh = np.empty((h_kv, L, d_h))
    st = _get().fp4o_dequant_seq(h_kv, d_h, fmt, 1 if rotate_k else 0, L, _p(k_src), _p(v_src),
                                 _p(kh), _p(vh))
    return kh, vh, int(st)


def fp4_decode_seq(q, k_src, v_src, *, fmt: int, sm_scale: float, rotate_k: bool = False):
    """Probe attention of one sequence: FP4-reconstructed bf16 K/V, fp64 softmax."""
    kh, vh, st = fp4_dequant_seq(k_src, v_src, fmt=fmt, rotate_k=rotate_k)
    out, lse = attend(q, kh, vh, sm_scale)
    return out, lse, st
