"""KV-concentration workload driver: continuous-refill and synchronous-wave
decode schedules over a pool of B slots (KV4-RL Sec. 4.1 and Prop. 4.1; App. C).

A response with prompt length P and generation length L ~ D (i.i.d.) occupies
one slot for L decode steps; at its age a (0 <= a < L) the slot's cached
context is P + a and the step appends the new token at position P + a, so the
decode attends over P + a + 1 positions.  The schedules differ only in when a
slot is refilled:

  continuous refill   a finished response is replaced before the next step
                      (every slot is busy at every step, B_t = B);
  synchronous waves   B responses start together and the wave ends when the
                      longest has finished (M_B = max L_i steps); a finished
                      slot idles until then.

The continuous-refill schedule can start in its stationary state: each slot's
current response length is drawn from the length-biased distribution
Pr(L* = l) = l Pr(L = l) / E[L] and its age uniformly from 0..l-1 (App. C
eq. A5), so that averages over a finite run carry no start-up transient.

`drive` runs a schedule through the library's C ABI on the GPU -- a prefill
append of each new response's first positions, one quantize-on-append per
active slot and one decode per step -- and measures the decode time; the
schedule's own step averages give the resident volume the kernels processed.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

from . import workloads as W


@dataclasses.dataclass
class Schedule:
    kind: str                 # "refill" or "waves"
    B: int
    P: int
    lens: np.ndarray          # int32 [D][B]: cache length after the step's append, 0 = idle
    resp: np.ndarray          # int32 [D][B]: response id in the slot (-1 = idle)
    prefill: List[np.ndarray]  # per step: int64 [k][3] rows (slot, response, positions to write)

    @property
    def steps(self) -> int:
        return int(self.lens.shape[0])

    def resident_context(self) -> np.ndarray:
        """Per step: sum over active slots of the cached context P + a before
        the step's append (the pages' l_i(t))."""
        act = self.lens > 0
        return np.where(act, self.lens - 1, 0).sum(axis=1)

    def active(self) -> np.ndarray:
        return (self.lens > 0).sum(axis=1)

    def averages(self) -> dict:
        """Step averages: resident context sum (volume / kappa), active slots,
        mean context of the active slots, and the tokens the decode reads."""
        act = self.active()
        ctx = self.resident_context()
        busy = act > 0
        return {"volume_tokens": float(ctx.mean()), "active": float(act.mean()),
                "mean_context": float(np.mean(ctx[busy] / act[busy])) if busy.any() else 0.0,
                "decode_tokens": float(self.lens.sum(axis=1).mean())}


def refill_schedule(B: int, P: int, support, pmf, steps: int, rng, stationary: bool = True):
    """Continuous refill for `steps` decode steps."""
    support = np.asarray(support, dtype=np.int64)
    pmf = np.asarray(pmf, dtype=np.float64)
    lens = np.zeros((steps, B), dtype=np.int32)
    resp = np.zeros((steps, B), dtype=np.int32)
    prefill: List[np.ndarray] = [np.zeros((0, 3), np.int64) for _ in range(steps)]
    if stationary:
        lb = support * pmf
        cur = support[rng.choice(len(support), size=B, p=lb / lb.sum())]
        age = (rng.random(B) * cur).astype(np.int64)          # uniform on 0..cur-1
    else:
        cur = W.sample_lengths(support, pmf, rng, B)
        age = np.zeros(B, dtype=np.int64)
    rid = np.arange(B, dtype=np.int64)
    nxt = B
    if steps:
        prefill[0] = np.stack([np.arange(B), rid, P + age], axis=1)   # prompt and earlier tokens
    for t in range(steps):
        lens[t] = P + age + 1
        resp[t] = rid
        age += 1
        done = np.nonzero(age == cur)[0]
        if len(done):
            cur[done] = W.sample_lengths(support, pmf, rng, len(done))
            age[done] = 0
            rid[done] = np.arange(nxt, nxt + len(done))
            nxt += len(done)
            if t + 1 < steps:
                prefill[t + 1] = np.stack([done, rid[done], np.full(len(done), P)], axis=1)
    return Schedule("refill", B, P, lens, resp, prefill)


def wave_schedule(B: int, P: int, support, pmf, waves: int, rng, max_steps: Optional[int] = None):
    """`waves` complete synchronous waves (cut at max_steps if given)."""
    blocks_l, blocks_r = [], []
    prefill: List[np.ndarray] = []
    nxt = 0
    for _ in range(waves):
        L = W.sample_lengths(support, pmf, rng, B)
        M = int(L.max())
        t = np.arange(M)[:, None]
        live = t < L[None, :]
        blocks_l.append(np.where(live, P + t + 1, 0).astype(np.int32))
        rid = np.arange(nxt, nxt + B, dtype=np.int64)
        blocks_r.append(np.where(live, rid[None, :], -1).astype(np.int32))
        prefill.append(np.stack([np.arange(B), rid, np.full(B, P)], axis=1))
        prefill.extend(np.zeros((0, 3), np.int64) for _ in range(M - 1))
        nxt += B
    lens = np.concatenate(blocks_l) if blocks_l else np.zeros((0, B), np.int32)
    resp = np.concatenate(blocks_r) if blocks_r else np.zeros((0, B), np.int32)
    if max_steps is not None:
        lens, resp, prefill = lens[:max_steps], resp[:max_steps], prefill[:max_steps]
    return Schedule("waves", B, P, lens, resp, prefill)


def decode_bytes(lens: np.ndarray, *, h_q: int, h_kv: int, d_h: int, group: int, sink: int,
                 recent: int) -> np.ndarray:
    """Algorithmic HBM bytes of one decode per row of `lens` (shape [..., B]):
    INT4 token-heads (codes + per-group Delta, m), INT8 token-heads (codes +
    fp16 scale), block-table entries of the INT4 pages, and the query read and
    output write of every active slot."""
    lens = np.asarray(lens, dtype=np.int64)
    n_p = np.minimum(lens, sink + recent)
    n_4 = lens - n_p
    int4_th = 2 * (d_h // 2 + 4 * (d_h // group))
    int8_th = 2 * (d_h + 2)
    per = h_kv * (n_p * int8_th + n_4 * int4_th) + ((lens + 15) // 16) * 4
    per = per + np.where(lens > 0, h_q * d_h * 2 * 2, 0)
    return per.sum(axis=-1)


def _sleep_cycles(us: float) -> int:
    return int(us * 2.1e3)   # at most the GB300 boost clock (2.07 GHz)


def _plan_chunk(sched: Schedule, c0: int, c1: int):
    """Host arrays for steps [c0, c1) of a driven schedule.

    rows  int64 [n]: token-pool rows of every K/V vector the chunk appends, in
          order: per step its prefill tokens, then its new tokens.
    ints  int32 [m]: per step six arrays, in order: prefill tok_seq, prefill
          tok_pos, prefill lengths [B], token tok_seq, token tok_pos, lengths
          after the step [B] (also the decode's seq_lens).
    plan  per step {"pre": (first row, count), "tok": (first row, count),
          "off": offsets of the six arrays in ints}."""
    B, P = sched.B, sched.P
    rows, ints, plan = [], [], []
    nrow = nint = 0
    for t in range(c0, c1):
        p_rows, p_seq, p_pos = [], [], []
        lens_pref = np.zeros(B, np.int32)
        for s_, r_, n_ in sched.prefill[t]:
            if n_ <= 0:
                continue
            pos = np.arange(n_, dtype=np.int64)
            p_rows.append(W.token_row(r_, pos))
            p_seq.append(np.full(n_, s_, np.int32))
            p_pos.append(pos.astype(np.int32))
            lens_pref[s_] = n_
        n_pre = int(sum(len(x) for x in p_seq))
        act = np.nonzero(sched.lens[t] > 0)[0]
        t_pos = (sched.lens[t, act] - 1).astype(np.int32)
        rows += p_rows + [W.token_row(sched.resp[t, act], t_pos)]
        seg = [np.concatenate(p_seq) if p_seq else np.zeros(0, np.int32),
               np.concatenate(p_pos) if p_pos else np.zeros(0, np.int32), lens_pref,
               act.astype(np.int32), t_pos, sched.lens[t].astype(np.int32)]
        off = [nint + sum(len(x) for x in seg[:k]) for k in range(6)]
        plan.append({"pre": (nrow, n_pre), "tok": (nrow + n_pre, len(act)), "off": off})
        ints += seg
        nint += sum(len(x) for x in seg)
        nrow += n_pre + len(act)
    rows = np.concatenate(rows).astype(np.int64) if rows else np.zeros(0, np.int64)
    ints = np.concatenate(ints).astype(np.int32) if ints else np.zeros(0, np.int32)
    assert len(rows) == nrow and len(ints) == nint
    return rows, ints, plan


def drive(sched: Schedule, *, h_q=32, h_kv=8, d_h=128, group=32, sink=4, recent=128, seed=0,
          device="cuda", chunk=32, gap_us=40.0, hadamard_k=False):
    """Run a schedule through the C ABI on one GPU.

    Per step: the prefill appends of responses that start (their first
    positions, multi-token kv4_quant_append), one kv4_quant_append of the new
    token of every active slot, and one kv4_decode_attn over all B slots
    (idle slots have length 0).  Token K/V and queries come from the seeded
    pools of workloads.py, indexed by (response, position).  Each timed call is
    preceded by a short GPU sleep so that its CUDA events bracket the kernels
    alone, not the host's launch latency.

    Returns the per-step decode, token-append and prefill times (ms), the
    outputs of the last step (bf16 out, fp32 lse, on the host) and the device
    status word."""
    import ctypes
    import torch
    from . import kv4
    from .cache import MixedKVCache
    B, P, D = sched.B, sched.P, sched.steps
    dev = torch.device(device)
    Lmax = max(1, int(sched.lens.max(initial=1)))
    mpps = (Lmax + 15) // 16
    cache = MixedKVCache(h_q=h_q, h_kv=h_kv, d_h=d_h, group=group, sink=sink, recent=recent,
                         max_seqs=B, num_pages=B * mpps, max_pages_per_seq=mpps, device=dev,
                         hadamard_k=hadamard_k)
    perm = np.random.default_rng([seed, 22]).permutation(B * mpps).astype(np.int32)
    cache.set_block_table(perm.reshape(B, mpps))
    kpool, vpool = W.token_pool(seed, h_kv, d_h)
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    Kp, Vp, Qp = to_dev(kpool), to_dev(vpool), to_dev(W.query_pool(seed, h_q, d_h))
    lib = kv4.load()
    lay = ctypes.byref(cache.layout)
    app_fn = lib.kv4_quant_append_hadamard if hadamard_k else lib.kv4_quant_append
    ws = cache.workspace(B)
    out = torch.empty((B, h_q, d_h), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, h_q), dtype=torch.float32, device=dev)
    qrot = torch.empty((B, h_q, d_h), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    scale = 1.0 / math.sqrt(d_h)
    row = h_kv * d_h * 2
    qbytes = B * h_q * d_h * 2
    gap = _sleep_cycles(gap_us)
    dec_ms = np.zeros(D)
    app_ms = np.zeros(D)
    pre_ms = np.zeros(D)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(chunk)]
    P_, bt, st = cache.paged.data_ptr(), cache.block_table.data_ptr(), cache.status.data_ptr()
    side = cache.side.data_ptr()

    def check(rc, what):
        if rc != kv4.KV4_OK:
            raise kv4.KV4Error(f"{what}: {lib.kv4_status_string(rc).decode()} (code {rc})")

    for c0 in range(0, D, chunk):
        c1 = min(D, c0 + chunk)
        rows, ints, plan = _plan_chunk(sched, c0, c1)
        nrow = len(rows)
        idx = torch.from_numpy(rows).to(dev)
        kbuf = torch.index_select(Kp, 0, idx) if nrow else Kp[:1]
        vbuf = torch.index_select(Vp, 0, idx) if nrow else Vp[:1]
        ib = torch.from_numpy(ints).to(dev)
        age = np.where(sched.lens[c0:c1] > 0, sched.lens[c0:c1] - 1 - P, 0)
        qidx = W.query_row(np.maximum(sched.resp[c0:c1], 0), np.maximum(age, 0)).reshape(-1)
        qbuf = torch.index_select(Qp, 0, torch.from_numpy(qidx).to(dev))
        kb, vb, ip, qb = kbuf.data_ptr(), vbuf.data_ptr(), ib.data_ptr(), qbuf.data_ptr()
        for i, ent in enumerate(plan):
            off = ent["off"]
            e = ev[i]
            torch.cuda._sleep(gap)
            e[0].record(stream)
            r0, n_pre = ent["pre"]
            if n_pre:
                check(app_fn(lay, P_, side, kb + r0 * row, vb + r0 * row, ip + 4 * off[0],
                             ip + 4 * off[1], n_pre, ip + 4 * off[2], bt, st, sp), "prefill append")
            e[1].record(stream)
            r1, n_tok = ent["tok"]
            if n_tok:
                check(app_fn(lay, P_, side, kb + r1 * row, vb + r1 * row, ip + 4 * off[3],
                             ip + 4 * off[4], n_tok, ip + 4 * off[5], bt, st, sp), "token append")
            e[2].record(stream)
            qptr = qb + i * qbytes
            if hadamard_k:   # the query side of the K rotation, outside the timed decode
                check(lib.kv4_hadamard_bf16(qptr, qrot.data_ptr(), B * h_q, d_h, sp), "query rotation")
                qptr = qrot.data_ptr()
            torch.cuda._sleep(gap)
            e[3].record(stream)
            check(lib.kv4_decode_attn(lay, P_, side, qptr, ip + 4 * off[5], B, bt, scale, 0,
                                      ws.data_ptr(), ws.numel(), out.data_ptr(), lse.data_ptr(),
                                      st, sp), "decode")
            e[4].record(stream)
        torch.cuda.synchronize(dev)
        for i in range(c1 - c0):
            pre_ms[c0 + i] = ev[i][0].elapsed_time(ev[i][1])
            app_ms[c0 + i] = ev[i][1].elapsed_time(ev[i][2])
            dec_ms[c0 + i] = ev[i][3].elapsed_time(ev[i][4])
        del kbuf, vbuf, qbuf, ib, idx
    return {"decode_ms": dec_ms, "append_ms": app_ms, "prefill_ms": pre_ms, "out": out.cpu(),
            "lse": lse.cpu(), "status": cache.read_status(), "cache": cache}


def slot_sources(sched: Schedule, t: int, b: int, *, h_q=32, h_kv=8, d_h=128, seed=0):
    """Host copies of what slot b holds at step t: source K and V (bf16 bits
    [h_kv][L][d_h], L = lens[t, b]) of its response, and that step's query
    (bf16 bits [h_q][d_h])."""
    L = int(sched.lens[t, b])
    r = int(sched.resp[t, b])
    kpool, vpool = W.token_pool(seed, h_kv, d_h)
    rows = W.token_row(r, np.arange(L))
    k = np.ascontiguousarray(kpool[rows].transpose(1, 0, 2))
    v = np.ascontiguousarray(vpool[rows].transpose(1, 0, 2))
    q = W.query_pool(seed, h_q, d_h)[W.query_row(r, L - 1 - sched.P)]
    return k, v, q


def report(sched: Schedule, res: dict, **shape) -> dict:
    """Step averages of a driven schedule: resident volume, occupancy, mean
    context, and the measured decode time and throughput."""
    avg = sched.averages()
    dec = res["decode_ms"]
    byt = decode_bytes(sched.lens, **shape)
    busy = sched.active() > 0
    return dict(avg, kind=sched.kind, steps=sched.steps, B=sched.B, P=sched.P,
                decode_ms_mean=float(dec.mean()), decode_ms_median=float(np.median(dec)),
                append_ms_mean=float(res["append_ms"].mean()),
                prefill_ms_total=float(res["prefill_ms"].sum()),
                decode_tokens_per_s=float(sched.lens.sum() / (dec.sum() / 1e3)),
                decode_GBps=float(byt.sum() / (dec.sum() / 1e3) / 1e9),
                decode_GBps_busy_steps=float(byt[busy].sum() / (dec[busy].sum() / 1e3) / 1e9)
                if busy.any() else 0.0,
                by_active=_by_active(sched.active(), sched.lens.sum(axis=1), byt, dec),
                status=int(res["status"]))


def _by_active(act, toks, byt, dec):
    """Decode time and bandwidth of the steps grouped by their active slots."""
    out = []
    for lo, hi in ((1, 8), (9, 32), (33, 128), (129, 1 << 30)):
        sel = (act >= lo) & (act <= hi)
        if sel.any():
            out.append({"active": f"{lo}-{hi}" if hi < (1 << 30) else f">={lo}", "steps": int(sel.sum()),
                        "tokens_mean": float(toks[sel].mean()), "decode_ms_mean": float(dec[sel].mean()),
                        "GBps": float(byt[sel].sum() / (dec[sel].sum() / 1e3) / 1e9)})
    return out
