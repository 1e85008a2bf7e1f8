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


class MixedKVCache:
    def __init__(self, *, h_q=32, h_kv=8, d_h=128, group=32, sink=4, recent=128, max_seqs,
                 num_pages, max_pages_per_seq, device="cuda", with_bf16=False):
        import torch
        self.layout = kv4.make_layout(h_q=h_q, h_kv=h_kv, d_h=d_h, group=group, sink=sink,
                                      recent=recent, max_seqs=max_seqs, num_pages=num_pages,
                                      max_pages_per_seq=max_pages_per_seq)
        rc = kv4.load().kv4_check_layout(__import__("ctypes").byref(self.layout))
        if rc != kv4.KV4_OK:
            raise kv4.KV4Error(f"bad layout: {kv4.load().kv4_status_string(rc).decode()}")
        self.device = torch.device(device)
        self.paged = torch.zeros(kv4.paged_cache_bytes(self.layout), dtype=torch.uint8,
                                 device=self.device)
        self.side = torch.zeros(max(16, kv4.side_cache_bytes(self.layout)), dtype=torch.uint8,
                                device=self.device)
        self.bf16 = (torch.zeros(kv4.bf16_cache_bytes(self.layout), dtype=torch.uint8,
                                 device=self.device) if with_bf16 else None)
        self.block_table = torch.full((max_seqs, max_pages_per_seq), -1, dtype=torch.int32,
                                      device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self._ws = {}

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.layout.head_dim)

    def set_block_table(self, bt):
        import torch
        bt = torch.as_tensor(np.asarray(bt, dtype=np.int32))
        self.block_table[: bt.shape[0], : bt.shape[1]].copy_(bt)

    def workspace(self, num_seqs: int, max_splits: int = 0):
        import torch
        key = (num_seqs, max_splits)
        if key not in self._ws:
            n = kv4.workspace_bytes(self.layout, num_seqs, max_splits)
            self._ws[key] = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
        return self._ws[key]

    def append(self, k_new, v_new, tok_seq, tok_pos, seq_lens, stream=None):
        kv4.kv4_quant_append(self.layout, self.paged, self.side, k_new, v_new, tok_seq, tok_pos,
                             seq_lens, self.block_table, self.status, stream)
        if self.bf16 is not None:
            kv4.kv4_bf16_append(self.layout, self.bf16, k_new, v_new, tok_seq, tok_pos, seq_lens,
                                self.block_table, self.status, stream)

    def decode(self, q, seq_lens, out, out_lse=None, max_splits=0, stream=None):
        ws = self.workspace(int(q.shape[0]), max_splits)
        kv4.kv4_decode_attn(self.layout, self.paged, self.side, q, seq_lens, self.block_table, ws,
                            out, out_lse, self.sm_scale, max_splits, self.status, stream)

    def decode_bf16(self, q, seq_lens, out, out_lse=None, max_splits=0, stream=None):
        ws = self.workspace(int(q.shape[0]), max_splits)
        kv4.kv4_bf16_decode_attn(self.layout, self.bf16, q, seq_lens, self.block_table, ws, out,
                                 out_lse, self.sm_scale, max_splits, self.status, stream)

    def read_status(self) -> int:
        return int(self.status.item())

    def clear_status(self):
        self.status.zero_()
