"""Seeded synthetic inputs for the KV4-RL decode path.

This module holds input generation only -- none of the method's arithmetic --
so that both the CUDA path (through the tests and the benchmark) and the CPU
oracle can be fed identical data.  Shapes follow the Qwen3-4B/8B and
Llama-3-8B attention layers the paper measures on (KV4-RL, Sec. 4.2 and
App. B.3-B.5: h_q = 32, h_kv = 8, d_h = 128, 16-token pages); the values are
N(0, 1) in bf16 with four fixed outlier key channels per kv head scaled by 8.
No dataset or checkpoint is involved: these inputs stand in for the paper's
rollout states.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

PAGE = 16
N_OUTLIER = 4
OUTLIER_GAIN = 8.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    h_q: int = 32
    h_kv: int = 8
    d_h: int = 128
    sink: int = 4
    recent: int = 128
    group: int = 32
    seed: int = 0
    lengths: str = "fixed"        # fixed | uniform | lognormal
    length: int = 512             # fixed length, or median for lognormal
    length_lo: int = 0
    length_hi: int = 0
    sigma: float = 0.0
    steps: int = 1
    layers: int = 1
    extra_pages: int = 0          # pool slack beyond the resident pages


WORKLOADS = {
    # Tiny single layer: 4 x 512, S=4, R=64, group 32, seed 1.
    "tiny_b4_l512": Workload("tiny_b4_l512", batch=4, sink=4, recent=64, group=32, seed=1,
                             lengths="fixed", length=512),
    # Qwen3-8B-shaped decode layer: batch 64, lengths U[1024, 8192], S=4, R=128.
    "qwen3_8b_b64": Workload("qwen3_8b_b64", batch=64, sink=4, recent=128, group=32, seed=2,
                             lengths="uniform", length_lo=1024, length_hi=8192),
    # Asynchronous-rollout concentration: batch 256, lognormal(median 3000,
    # sigma 0.8) clipped to [256, 16384], 100 append+decode steps.
    "rollout_b256": Workload("rollout_b256", batch=256, sink=4, recent=128, group=32, seed=3,
                             lengths="lognormal", length=3000, sigma=0.8, length_lo=256,
                             length_hi=16384, steps=100),
    # Long-context single request: 1 x 131072, S=4, R=256.
    "long_128k": Workload("long_128k", batch=1, sink=4, recent=256, group=32, seed=4,
                          lengths="fixed", length=131072),
    # 36-layer Qwen3-8B-shaped step: 128 x 8192 per layer, seed 500+layer.
    "qwen3_8b_36l": Workload("qwen3_8b_36l", batch=128, sink=4, recent=128, group=32, seed=500,
                             lengths="fixed", length=8192, layers=36),
}


def seq_lengths(w: Workload) -> np.ndarray:
    """Context lengths L_b (positions in the cache after the decode step's append)."""
    rng = np.random.default_rng([w.seed, 1])
    if w.lengths == "fixed":
        return np.full((w.batch,), w.length, dtype=np.int32)
    if w.lengths == "uniform":
        return rng.integers(w.length_lo, w.length_hi + 1, size=w.batch).astype(np.int32)
    if w.lengths == "lognormal":
        x = np.exp(rng.normal(math.log(w.length), w.sigma, size=w.batch))
        return np.clip(np.round(x), w.length_lo, w.length_hi).astype(np.int32)
    raise ValueError(w.lengths)


def lognormal_length_pmf(median: float, sigma: float, lo: int, hi: int):
    """The exact distribution of the lognormal lengths seq_lengths draws:
    round(exp(N(log median, sigma^2))) clipped to [lo, hi].  Returns (support,
    pmf) over lo..hi; the clipped tails sit on lo and hi."""
    l = np.arange(lo, hi + 1, dtype=np.float64)
    mu = math.log(median)
    cdf = lambda x: 0.5 * (1.0 + np.vectorize(math.erf)((np.log(x) - mu) / (sigma * math.sqrt(2.0))))
    upper = np.append(cdf(l[:-1] + 0.5), 1.0)
    lower = np.concatenate([[0.0], cdf(l[1:] - 0.5)])
    pmf = np.maximum(upper - lower, 0.0)
    return l.astype(np.int64), pmf / pmf.sum()


def sample_lengths(support, pmf, rng, n: int) -> np.ndarray:
    """n i.i.d. lengths from an explicit pmf."""
    return np.asarray(support)[rng.choice(len(support), size=n, p=pmf)].astype(np.int64)


def outlier_channels(seed: int, h_kv: int, d_h: int) -> np.ndarray:
    """Four fixed key channels per kv head, drawn once per seed: int32 [h_kv][4]."""
    rng = np.random.default_rng([seed, 2])
    return np.stack([rng.choice(d_h, size=N_OUTLIER, replace=False) for _ in range(h_kv)]).astype(np.int32)


def block_table(seed: int, lens: np.ndarray, max_pages_per_seq: int, num_pages: int) -> np.ndarray:
    """Seeded permutation of the page pool handed out to the sequences in order.
    Unused entries are -1.  int32 [B][max_pages_per_seq]."""
    rng = np.random.default_rng([seed, 3])
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((len(lens), max_pages_per_seq), -1, dtype=np.int32)
    k = 0
    for b, L in enumerate(lens):
        n = (int(L) + PAGE - 1) // PAGE
        bt[b, :n] = perm[k:k + n]
        k += n
    assert k <= num_pages
    return bt


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (input preparation)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def kv_numpy(seed: int, seq: int, h_kv: int, L: int, d_h: int, outl: np.ndarray, p0: int = 0):
    """Source K and V of positions [p0, L) of sequence ``seq``: bf16 bits
    [h_kv][L-p0][d_h].  Keys carry the outlier channels.  Each position's
    values depend only on (seed, seq, position), so any window can be
    regenerated on its own."""
    n = L - p0
    K = np.empty((h_kv, n, d_h), dtype=np.float32)
    V = np.empty((h_kv, n, d_h), dtype=np.float32)
    for i, p in enumerate(range(p0, L)):
        rng = np.random.default_rng([seed, 10, seq, p])
        kv = rng.standard_normal((2, h_kv, d_h), dtype=np.float32)
        K[:, i, :] = kv[0]
        V[:, i, :] = kv[1]
    for h in range(h_kv):
        K[h][:, outl[h]] *= OUTLIER_GAIN
    return f32_to_bf16_bits(K), f32_to_bf16_bits(V)


def kv_numpy_block(seed: int, seq: int, h_kv: int, L: int, d_h: int, outl: np.ndarray):
    """Faster whole-sequence variant (one generator per sequence) for positions
    [0, L): bf16 bits [h_kv][L][d_h]."""
    rng = np.random.default_rng([seed, 11, seq])
    K = rng.standard_normal((h_kv, L, d_h), dtype=np.float32)
    V = rng.standard_normal((h_kv, L, d_h), dtype=np.float32)
    for h in range(h_kv):
        K[h][:, outl[h]] *= OUTLIER_GAIN
    return f32_to_bf16_bits(K), f32_to_bf16_bits(V)


def q_numpy(seed: int, B: int, h_q: int, d_h: int, step: int = 0) -> np.ndarray:
    rng = np.random.default_rng([seed, 12, step])
    return f32_to_bf16_bits(rng.standard_normal((B, h_q, d_h), dtype=np.float32))


# ------------------------------------------------- rollout token content

# Rollout drivers draw every token's K/V and every step's query from fixed
# seeded pools, indexed by (response id, position), so that any slot's cache
# contents can be regenerated on the host for a parity check.
POOL_TOKENS = 4099
POOL_QUERIES = 1031


def token_pool(seed: int, h_kv: int, d_h: int, n: int = POOL_TOKENS):
    """K and V rows of the pool: bf16 bits [n][h_kv][d_h], keys with the
    outlier channels of this seed."""
    rng = np.random.default_rng([seed, 20])
    K = rng.standard_normal((n, h_kv, d_h), dtype=np.float32)
    V = rng.standard_normal((n, h_kv, d_h), dtype=np.float32)
    outl = outlier_channels(seed, h_kv, d_h)
    for h in range(h_kv):
        K[:, h, outl[h]] *= OUTLIER_GAIN
    return f32_to_bf16_bits(K), f32_to_bf16_bits(V)


def query_pool(seed: int, h_q: int, d_h: int, n: int = POOL_QUERIES) -> np.ndarray:
    rng = np.random.default_rng([seed, 21])
    return f32_to_bf16_bits(rng.standard_normal((n, h_q, d_h), dtype=np.float32))


def token_row(resp, pos, n: int = POOL_TOKENS):
    """Pool row of the token at position ``pos`` of response ``resp``."""
    return (np.asarray(resp, dtype=np.int64) * 7919 + np.asarray(pos, dtype=np.int64)) % n


def query_row(resp, age, n: int = POOL_QUERIES):
    """Pool row of the query of response ``resp`` at decode step ``age``."""
    return (np.asarray(resp, dtype=np.int64) * 131 + np.asarray(age, dtype=np.int64)) % n


# ----------------------------------------------------------- device variants

def torch_generator(seed: int, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def kv_torch(gen, h_kv: int, n: int, d_h: int, outl: np.ndarray, device):
    """Device-side K/V source for n positions: bf16 [n][h_kv][d_h] each (token-major,
    the layout the append entry point reads)."""
    import torch
    K = torch.randn((n, h_kv, d_h), generator=gen, device=device, dtype=torch.float32)
    V = torch.randn((n, h_kv, d_h), generator=gen, device=device, dtype=torch.float32)
    idx = torch.as_tensor(outl, device=device, dtype=torch.long)
    for h in range(h_kv):
        K[:, h, idx[h]] *= OUTLIER_GAIN
    return K.to(torch.bfloat16), V.to(torch.bfloat16)


def pool_pages(lens: np.ndarray, extra: int = 0) -> int:
    return int(sum((int(L) + PAGE - 1) // PAGE for L in lens)) + int(extra)


def describe(w: Workload) -> dict:
    lens = seq_lengths(w)
    return {"workload": w.name, "batch": w.batch, "h_q": w.h_q, "h_kv": w.h_kv, "d_h": w.d_h,
            "sink": w.sink, "recent": w.recent, "group": w.group, "seed": w.seed,
            "mean_len": float(lens.mean()), "total_tokens": int(lens.sum())}


def sample_rows(seed: int, n_total: int, n_pick: int, extra: Optional[list] = None) -> np.ndarray:
    """Seeded sample of sequence indices used for full-size parity checks."""
    rng = np.random.default_rng([seed, 13])
    pick = set(rng.choice(n_total, size=min(n_pick, n_total), replace=False).tolist())
    if extra:
        pick.update(int(e) for e in extra if 0 <= int(e) < n_total)
    return np.array(sorted(pick), dtype=np.int64)
