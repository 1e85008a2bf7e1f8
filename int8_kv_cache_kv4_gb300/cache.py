"""Device-resident mixed INT4/INT8 paged KV cache of one attention layer.

A small convenience wrapper: PyTorch allocates the caller-owned buffers that
the C ABI sizes (paged INT4 pool, INT8 side cache, block table, workspace),
and the methods forward to the binding.  No compute happens here.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

from . import kv4
from . import workloads as W


class _LayerCache:
    """What both cache kinds share: the layout, block table, status word,
    per-shape workspaces and the rotated-query scratch."""

    def _init_common(self, layout, max_seqs, max_pages_per_seq, device, hadamard_k):
        import torch
        import ctypes
        rc = kv4.load().kv4_check_layout(ctypes.byref(layout))
        if rc != kv4.KV4_OK:
            raise kv4.KV4Error(f"bad layout: {kv4.load().kv4_status_string(rc).decode()}")
        self.layout = layout
        self.device = torch.device(device)
        self.block_table = torch.full((max_seqs, max_pages_per_seq), -1, dtype=torch.int32,
                                      device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.hadamard_k = bool(hadamard_k)
        self._ws = {}
        self._qrot = {}

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.layout.head_dim)

    def set_block_table(self, bt):
        import torch
        bt = torch.as_tensor(np.asarray(bt, dtype=np.int32))
        self.block_table[: bt.shape[0], : bt.shape[1]].copy_(bt)

    def workspace(self, num_seqs: int, max_splits: int = 0, bf16: bool = False):
        import torch
        key = (num_seqs, max_splits, bf16)
        if key not in self._ws:
            n = (kv4.bf16_workspace_bytes if bf16 else kv4.workspace_bytes)(self.layout, num_seqs,
                                                                             max_splits)
            self._ws[key] = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
        return self._ws[key]

    def rotated_query(self, q, stream=None):
        """q rotated like the stored keys (a scratch tensor reused per shape)."""
        import torch
        key = tuple(q.shape)
        if key not in self._qrot:
            self._qrot[key] = torch.empty_like(q)
        return kv4.kv4_hadamard_bf16(q, self._qrot[key], stream)

    def read_status(self) -> int:
        return int(self.status.item())

    def clear_status(self):
        self.status.zero_()


class MixedKVCache(_LayerCache):
    """The mixed INT4/INT8 cache.  hadamard_k=True stores K rotated by the
    normalized Hadamard matrix (kv4_quant_append_hadamard) and rotates each
    query the same way (kv4_hadamard_bf16) before decode; callers pass
    unrotated K and q.  with_bf16 keeps an unquantized comparator copy."""

    def __init__(self, *, h_q=32, h_kv=8, d_h=128, group=32, sink=4, recent=128, max_seqs,
                 num_pages, max_pages_per_seq, device="cuda", with_bf16=False, hadamard_k=False):
        import torch
        layout = kv4.make_layout(h_q=h_q, h_kv=h_kv, d_h=d_h, group=group, sink=sink,
                                 recent=recent, max_seqs=max_seqs, num_pages=num_pages,
                                 max_pages_per_seq=max_pages_per_seq)
        self._init_common(layout, max_seqs, max_pages_per_seq, device, hadamard_k)
        self.paged = torch.zeros(kv4.paged_cache_bytes(self.layout), dtype=torch.uint8,
                                 device=self.device)
        self.side = torch.zeros(max(16, kv4.side_cache_bytes(self.layout)), dtype=torch.uint8,
                                device=self.device)
        self.bf16 = (torch.zeros(kv4.bf16_cache_bytes(self.layout), dtype=torch.uint8,
                                 device=self.device) if with_bf16 else None)

    def append(self, k_new, v_new, tok_seq, tok_pos, seq_lens, stream=None, comparator=True):
        """kv4_quant_append (or its Hadamard form); with comparator=True also
        the bf16 comparator cache, when this cache keeps one."""
        fn = kv4.kv4_quant_append_hadamard if self.hadamard_k else kv4.kv4_quant_append
        fn(self.layout, self.paged, self.side, k_new, v_new, tok_seq, tok_pos, seq_lens,
           self.block_table, self.status, stream)
        if comparator and self.bf16 is not None:
            kv4.kv4_bf16_append(self.layout, self.bf16, k_new, v_new, tok_seq, tok_pos, seq_lens,
                                self.block_table, self.status, stream)

    def decode(self, q, seq_lens, out, out_lse=None, max_splits=0, stream=None,
               separate_rotation=False):
        """Decode of q against this cache.  With the Hadamard K-rotation the
        query is rotated by the decode call itself (kv4_decode_attn_hadamard);
        separate_rotation=True rotates it first with kv4_hadamard_bf16 into a
        scratch buffer and calls kv4_decode_attn (same result, one more
        launch)."""
        ws = self.workspace(int(q.shape[0]), max_splits)
        rotate = self.hadamard_k
        if rotate and separate_rotation:
            q = self.rotated_query(q, stream)
            rotate = False
        kv4.kv4_decode_attn(self.layout, self.paged, self.side, q, seq_lens, self.block_table, ws,
                            out, out_lse, self.sm_scale, max_splits, self.status, stream,
                            rotate_q=rotate)

    def decode_bf16(self, q, seq_lens, out, out_lse=None, max_splits=0, stream=None):
        ws = self.workspace(int(q.shape[0]), max_splits, bf16=True)
        kv4.kv4_bf16_decode_attn(self.layout, self.bf16, q, seq_lens, self.block_table, ws, out,
                                 out_lse, self.sm_scale, max_splits, self.status, stream)


class FP4ProbeCache(_LayerCache):
    """FP4 probe cache of one layer (KV4-RL App. D.4: NVFP4 or MXFP4 K/V,
    reconstructed and attended with bf16 operands).  `append` writes the
    packed format; `decode` reconstructs the pool into a bf16 comparator cache
    and runs the bf16 decode over it, rotating the query when K is rotated.
    Same call shapes as MixedKVCache.  No compute happens here."""

    def __init__(self, *, fmt, h_q=32, h_kv=8, d_h=128, max_seqs, num_pages, max_pages_per_seq,
                 device="cuda", hadamard_k=False):
        import torch
        self.fmt = int(fmt)
        layout = kv4.make_layout(h_q=h_q, h_kv=h_kv, d_h=d_h, group=32, sink=0, recent=0,
                                 max_seqs=max_seqs, num_pages=num_pages,
                                 max_pages_per_seq=max_pages_per_seq)
        self._init_common(layout, max_seqs, max_pages_per_seq, device, hadamard_k)
        self.cache = torch.zeros(kv4.fp4_cache_bytes(self.layout), dtype=torch.uint8,
                                 device=self.device)
        self.bf16 = torch.zeros(kv4.bf16_cache_bytes(self.layout), dtype=torch.uint8,
                                device=self.device)

    def append(self, k_new, v_new, tok_seq, tok_pos, seq_lens, stream=None):
        kv4.kv4_fp4_append(self.layout, self.fmt, self.cache, k_new, v_new, tok_seq, tok_pos,
                           seq_lens, self.block_table, self.hadamard_k, self.status, stream)

    def reconstruct(self, stream=None):
        kv4.kv4_fp4_to_bf16(self.layout, self.fmt, self.cache, self.bf16, stream)

    def decode(self, q, seq_lens, out, out_lse=None, max_splits=0, stream=None):
        self.reconstruct(stream)
        if self.hadamard_k:
            q = self.rotated_query(q, stream)
        ws = self.workspace(int(q.shape[0]), max_splits, bf16=True)
        kv4.kv4_bf16_decode_attn(self.layout, self.bf16, q, seq_lens, self.block_table, ws, out,
                                 out_lse, self.sm_scale, max_splits, self.status, stream)


def build_workload(w, dev, with_bf16=False, lens=None, group=None, recent=None, seed=None,
                   extra_tokens=0, hadamard_k=False, fp4=None):
    """Populate a cache with a seeded synthetic workload (see workloads.py):
    positions [0, L-1) of every sequence by bulk appends, then return the
    decode step's inputs (the new token at position L-1 and the query).
    Sequence b's source K/V come from the generator seeded seed*1000003+b, the
    step token and query from seed*1000003+999983, so any sequence can be
    regenerated for a parity check.  `extra_tokens` reserves block-table room
    for that many later appends per sequence.  hadamard_k: the cache stores
    rotated K (MixedKVCache(hadamard_k=True)).  fp4: KV4_FP4_NVFP4 or
    KV4_FP4_MXFP4 builds an FP4ProbeCache of that format instead."""
    import torch
    import dataclasses
    if group is not None or recent is not None or seed is not None:
        w = dataclasses.replace(w, group=w.group if group is None else group,
                                recent=w.recent if recent is None else recent,
                                seed=w.seed if seed is None else seed)
    lens = W.seq_lengths(w) if lens is None else lens
    B = len(lens)
    cap = lens + int(extra_tokens)
    mpps = (int(cap.max()) + 15) // 16
    num_pages = W.pool_pages(cap, w.extra_pages)
    if fp4:
        cache = FP4ProbeCache(fmt=fp4, h_q=w.h_q, h_kv=w.h_kv, d_h=w.d_h, max_seqs=B,
                              num_pages=num_pages, max_pages_per_seq=mpps, device=dev,
                              hadamard_k=hadamard_k)
    else:
        cache = MixedKVCache(h_q=w.h_q, h_kv=w.h_kv, d_h=w.d_h, group=w.group, sink=w.sink,
                             recent=w.recent, max_seqs=B, num_pages=num_pages,
                             max_pages_per_seq=mpps, device=dev, with_bf16=with_bf16,
                             hadamard_k=hadamard_k)
    cache.set_block_table(W.block_table(w.seed, cap, mpps, num_pages))
    outl = W.outlier_channels(w.seed, w.h_kv, w.d_h)
    # populate positions [0, L-1) of every sequence (prefill-style bulk append)
    for b, L in enumerate(lens):
        n = int(L) - 1
        if n <= 0:
            continue
        gen = W.torch_generator(w.seed * 1000003 + b, dev)
        k, v = W.kv_torch(gen, w.h_kv, n, w.d_h, outl, dev)
        seq = torch.full((n,), b, dtype=torch.int32, device=dev)
        pos = torch.arange(n, dtype=torch.int32, device=dev)
        lens_now = torch.as_tensor(np.maximum(lens - 1, 0).astype(np.int32), device=dev)
        cache.append(k, v, seq, pos, lens_now)
    # the step's new token (position L-1) and query
    k_new, v_new, q = step_inputs(w, B, 0, dev)
    step = {
        "k": k_new, "v": v_new, "q": q,
        "seq": torch.arange(B, dtype=torch.int32, device=dev),
        "pos": torch.as_tensor((lens - 1).astype(np.int32), device=dev),
        "lens": torch.as_tensor(lens.astype(np.int32), device=dev),
        "out": torch.empty((B, w.h_q, w.d_h), dtype=torch.bfloat16, device=dev),
        "lse": torch.empty((B, w.h_q), dtype=torch.float32, device=dev),
    }
    torch.cuda.synchronize()
    return cache, step, lens, w


def step_inputs(w, B, step, dev):
    """New K/V token of every sequence and the query for rollout step `step`
    (step 0 is the token build_workload returns)."""
    import torch
    gen = W.torch_generator(w.seed * 1000003 + 999983 + 7919 * step, dev)
    outl = W.outlier_channels(w.seed, w.h_kv, w.d_h)
    k_new, v_new = W.kv_torch(gen, w.h_kv, B, w.d_h, outl, dev)
    q = torch.randn((B, w.h_q, w.d_h), generator=gen, device=dev).to(torch.bfloat16)
    return k_new, v_new, q


def source_kv(w, b, L0, dev, steps=1):
    """Regenerate the source K/V of sequence b (bf16 bits, numpy
    [h_kv][L0 - 1 + steps][d_h]): the populated prefix [0, L0 - 1) and one
    token per rollout step."""
    import torch
    outl = W.outlier_channels(w.seed, w.h_kv, w.d_h)
    parts_k, parts_v = [], []
    n = int(L0) - 1
    if n > 0:
        gen = W.torch_generator(w.seed * 1000003 + b, dev)
        k, v = W.kv_torch(gen, w.h_kv, n, w.d_h, outl, dev)
        parts_k.append(k)
        parts_v.append(v)
    B = None
    for s in range(steps):
        kk, vv, _ = step_inputs(w, w.batch, s, dev)
        parts_k.append(kk[b:b + 1])
        parts_v.append(vv[b:b + 1])
    k = torch.cat(parts_k).transpose(0, 1).contiguous()
    v = torch.cat(parts_v).transpose(0, 1).contiguous()
    return (k.view(torch.int16).cpu().numpy().view(np.uint16),
            v.view(torch.int16).cpu().numpy().view(np.uint16))
