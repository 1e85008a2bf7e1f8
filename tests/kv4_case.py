"""Shared helpers for the GPU parity tests: build one seeded case, run the
CUDA path through the C ABI and the CPU oracle on the same inputs."""
from __future__ import annotations

import math

import numpy as np

import oracle
from int8_kv_cache_kv4_gb300 import workloads as W

# stated tolerance for bf16 attention outputs against the fp64 oracle
MAX_ABS = 2e-3
MEAN_ABS = 2e-4
LSE_ABS = 1e-3   # fp32 scores and normaliser vs fp64


def scale_bf16(bits, e):
    """bf16 values (bit patterns) times 2^e: exact while the results stay in
    bf16's normal range (checked)."""
    if e == 0:
        return bits
    x = W.bf16_bits_to_f32(bits) * np.float32(2.0 ** e)
    out = W.f32_to_bf16_bits(x)
    assert np.array_equal(W.bf16_bits_to_f32(out), x), "scaling left bf16's exact range"
    return out


class Case:
    """A batch of sequences with seeded K/V/q, a seeded page permutation and
    token lists for a populate append followed by a one-token append."""

    def __init__(self, lens, *, h_q=32, h_kv=8, d_h=128, g=32, S=4, R=64, seed=1, extra_pages=3,
                 rotate_k=False, k_exp=0, v_exp=0, q_exp=0):
        self.rotate_k = bool(rotate_k)
        self.lens = np.asarray(lens, dtype=np.int32)
        self.B = len(self.lens)
        self.h_q, self.h_kv, self.d_h, self.g, self.S, self.R = h_q, h_kv, d_h, g, S, R
        self.seed = seed
        self.mpps = max(1, (int(self.lens.max(initial=0)) + 15) // 16)
        self.num_pages = W.pool_pages(self.lens, extra_pages)
        self.bt = W.block_table(seed, self.lens, self.mpps, self.num_pages)
        outl = W.outlier_channels(seed, h_kv, d_h)
        self.k = []
        self.v = []
        for b, L in enumerate(self.lens):
            kb, vb = W.kv_numpy_block(seed, b, h_kv, int(L), d_h, outl)
            self.k.append(scale_bf16(kb, k_exp))
            self.v.append(scale_bf16(vb, v_exp))
        self.q = scale_bf16(W.q_numpy(seed, self.B, h_q, d_h), q_exp)
        self.sm_scale = 1.0 / math.sqrt(d_h)

    def layout_kw(self):
        return dict(h_kv=self.h_kv, d_h=self.d_h, g=self.g, S=self.S, R=self.R, max_seqs=self.B,
                    num_pages=self.num_pages, max_pages_per_seq=self.mpps)

    def tokens(self, stage):
        """stage 0: positions [0, L-1) of every sequence; stage 1: position L-1.
        Returns (k [T][h_kv][d_h], v, tok_seq, tok_pos, seq_lens_after)."""
        ks, vs, seqs, poss = [], [], [], []
        for b, L in enumerate(self.lens):
            L = int(L)
            rng = range(0, max(L - 1, 0)) if stage == 0 else (range(L - 1, L) if L > 0 else range(0))
            for p in rng:
                ks.append(self.k[b][:, p, :])
                vs.append(self.v[b][:, p, :])
                seqs.append(b)
                poss.append(p)
        lens_after = np.maximum(self.lens - (1 if stage == 0 else 0), 0).astype(np.int32)
        if not ks:
            z = np.zeros((0, self.h_kv, self.d_h), dtype=np.uint16)
            return z, z, np.zeros(0, np.int32), np.zeros(0, np.int32), lens_after
        return (np.ascontiguousarray(np.stack(ks)), np.ascontiguousarray(np.stack(vs)),
                np.array(seqs, np.int32), np.array(poss, np.int32), lens_after)

    # ------------------------------------------------------------- oracle
    def oracle_cache(self):
        paged = np.zeros(self.num_pages * self.h_kv * oracle.chunk_bytes(self.d_h, self.g), np.uint8)
        side = np.zeros(max(16, self.B * self.h_kv * oracle.side_block_bytes(self.d_h, self.S, self.R)),
                        np.uint8)
        st = 0
        for stage in (0, 1):
            k, v, s, p, la = self.tokens(stage)
            st |= oracle.quant_append(**self.layout_kw(), paged=paged, side=side, k_new=k, v_new=v,
                                      tok_seq=s, tok_pos=p, seq_lens=la, block_table=self.bt,
                                      rotate_k=self.rotate_k)
        return paged, side, st

    def oracle_decode(self, seqs=None):
        seqs = range(self.B) if seqs is None else seqs
        outs, lses = {}, {}
        for b in seqs:
            q = oracle.hadamard_bf16(self.q[b]) if self.rotate_k else self.q[b]
            o, l, _ = oracle.decode_seq(q, self.k[b], self.v[b], g=self.g, S=self.S,
                                        R=self.R, sm_scale=self.sm_scale, rotate_k=self.rotate_k)
            outs[b], lses[b] = o, l
        return outs, lses

    def oracle_bf16(self, seqs=None):
        seqs = range(self.B) if seqs is None else seqs
        outs, lses = {}, {}
        for b in seqs:
            kh = W.bf16_bits_to_f32(self.k[b]).astype(np.float64)
            vh = W.bf16_bits_to_f32(self.v[b]).astype(np.float64)
            outs[b], lses[b] = oracle.attend(self.q[b], kh, vh, self.sm_scale)
        return outs, lses

    # ---------------------------------------------------------------- GPU
    def gpu(self, *, with_bf16=False):
        import torch
        from int8_kv_cache_kv4_gb300.cache import MixedKVCache
        dev = torch.device("cuda")
        c = MixedKVCache(h_q=self.h_q, h_kv=self.h_kv, d_h=self.d_h, group=self.g, sink=self.S,
                         recent=self.R, max_seqs=self.B, num_pages=self.num_pages,
                         max_pages_per_seq=self.mpps, device=dev, with_bf16=with_bf16,
                         hadamard_k=self.rotate_k)
        c.set_block_table(self.bt)
        for stage in (0, 1):
            k, v, s, p, la = self.tokens(stage)
            if len(s) == 0:
                continue
            to = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev).view(dt)
            c.append(to(k, torch.int16).view(torch.bfloat16), to(v, torch.int16).view(torch.bfloat16),
                     to(s, torch.int32), to(p, torch.int32), to(la, torch.int32))
        return c

    def gpu_decode(self, c, max_splits=0, bf16=False):
        import torch
        dev = c.device
        q = torch.from_numpy(self.q.view(np.int16)).to(dev).view(torch.bfloat16)
        lens = torch.from_numpy(self.lens).to(dev)
        out = torch.empty((self.B, self.h_q, self.d_h), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((self.B, self.h_q), dtype=torch.float32, device=dev)
        if bf16:
            c.decode_bf16(q, lens, out, lse, max_splits=max_splits)
        else:
            c.decode(q, lens, out, lse, max_splits=max_splits)
        torch.cuda.synchronize()
        return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def half_ulp_bf16(x):
    """Half a bf16 ulp at |x|: the rounding error any bf16 output must carry."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def ulp_bf16(x):
    """One bf16 ulp at |x| (8 significant bits)."""
    return 2.0 * half_ulp_bf16(x)


def oracle_decode_many(jobs, threads=None):
    """oracle.decode_seq over many sequences on the host's cores.  jobs:
    {key: (q, k_src, v_src, kwargs)}.  The oracle is C behind ctypes, which
    releases the GIL during each call, so threads run the sequences in
    parallel without copying their sources."""
    import concurrent.futures as cf
    import os
    threads = threads or min(len(jobs), os.cpu_count() or 1) or 1

    def one(item):
        key, (q, k, v, kw) = item
        o, l, st = oracle.decode_seq(q, k, v, **kw)
        assert st == 0
        return key, o, l

    outs, lses = {}, {}
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        for key, o, l in ex.map(one, list(jobs.items())):
            outs[key], lses[key] = o, l
    return outs, lses


def compare_outputs(out, lse, ref_out, ref_lse, seqs, lens, max_abs=MAX_ABS, mean_abs=MEAN_ABS,
                    label=""):
    """bf16 decode outputs against the fp64 oracle, with the raw error
    e = |out - ref|.

    - Every element: e <= 2e-3, or, where |ref| >= 0.5 (half a bf16 ulp there
      is 2^-9 or more, so the output's own rounding alone can reach 2e-3),
      `out` is one of the two bf16 values bracketing ref (e < 1 ulp: faithful
      rounding).  Below 0.5 the second clause adds nothing: an ulp there is
      at most 2^-9 < 2e-3.
    - Mean: when max |ref| < 0.5 over the compared sequences (every
      long-context and full-size workload), the raw mean e <= 2e-4 and the raw
      max e <= 2e-3, the stated figures as they stand.  Otherwise the mean of
      |out - bf16(ref)|, the deviation from the correctly rounded oracle
      output, is <= 2e-4 (the raw mean of such a case is dominated by the
      rounding of the |o| >= 0.5 outputs, which no bf16 output avoids).
    The log-normaliser (fp32) is within 1e-3 of the oracle's.
    Returns (raw max, raw mean) and prints both statistics."""
    raws, rnds, refs = [], [], []
    for b in seqs:
        if int(lens[b]) == 0:
            assert np.all(out[b] == 0), f"seq {b}: empty sequence must give zeros"
            assert np.all(np.isneginf(lse[b]))
            continue
        ref = np.asarray(ref_out[b], dtype=np.float64)
        e = np.abs(out[b] - ref)
        ok = (e <= max_abs) | ((np.abs(ref) >= 0.5) & (e < ulp_bf16(ref)))
        assert ok.all(), (f"seq {b}: {int((~ok).sum())} outputs beyond 2e-3 and not a bf16 "
                          f"neighbour of the oracle value (worst {e[~ok].max():.3e})")
        raws.append(e.ravel())
        rnds.append(np.abs(out[b] - oracle.bf16_round(ref)).ravel())
        refs.append(np.abs(ref).ravel())
        np.testing.assert_allclose(lse[b], ref_lse[b], atol=LSE_ABS, rtol=0,
                                   err_msg=f"lse of seq {b}")
    if not raws:
        return 0.0, 0.0
    raw = np.concatenate(raws)
    rnd = np.concatenate(rnds)
    big = float(np.concatenate(refs).max())
    print(f"{label} raw max {raw.max():.3e} raw mean {raw.mean():.3e} | vs bf16(oracle): max "
          f"{rnd.max():.3e} mean {rnd.mean():.3e} | max |o| {big:.3f}")
    if big < 0.5:
        assert raw.max() <= max_abs, f"raw max abs err {raw.max():.3e} > {max_abs}"
        assert raw.mean() <= mean_abs, f"raw mean abs err {raw.mean():.3e} > {mean_abs}"
    else:
        assert rnd.mean() <= mean_abs, f"mean |out - bf16(ref)| {rnd.mean():.3e} > {mean_abs}"
    return float(raw.max()), float(raw.mean())
