#!/usr/bin/env python
"""Benchmark of the KV4-RL decode hot path on GB300.

One step = the whole hot path over one batch: quantize-on-append of one new
K/V token per sequence (kv4_quant_append) followed by mixed INT4/INT8 split-KV
decode attention with the eq. A1 merge (kv4_decode_attn).  The default
workload is the Qwen3-8B-shaped decode layer: 64 sequences with lengths
uniform in [1024, 8192], h_q=32, h_kv=8, d_h=128, S=4, R=128, group 32,
shuffled 16-token pages, seeded synthetic bf16 K/V/q (4 outlier key channels
per kv head scaled by 8).  The cache (~385 MB) is larger than L2, so every
step streams it from HBM.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from int8_kv_cache_kv4_gb300 import workloads as W  # noqa: E402
from int8_kv_cache_kv4_gb300.cache import build_workload  # noqa: E402

METRIC = "decode-attn resident KV tokens/s per layer and achieved HBM GB/s vs 8 TB/s"
UNIT = "tokens/s"
# seed offset of the second layer cache the timed steps alternate with
SECOND_LAYER_SEED = 100

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the default decode kernel on the default workload, from the ncu capture
# summarised in profiles/decode_stream_kernel_qwen3_8b_b64.md and
# profiles/launch_list_long_128k.md.  Keyed by a
# hash of the sources that kernel is compiled from: once they change, the
# figure no longer describes the kernel and the bench reports null.
KERNEL_SOURCES = ["kv4_decode_stream.cu", "kv4_stream_common.cuh", "kv4_mma.cuh", "kv4_decode_common.cuh",
                  "kv4_common.cuh"]
TRAFFIC = {("153be8b4d64b8801", "qwen3_8b_b64"): 387799808 + 1533440,
           ("153be8b4d64b8801", "long_128k"): 168165632 + 687616}


# ------------------------------------------------------------------ helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "int8_kv_cache_kv4_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def algorithmic_bytes(lens, w: W.Workload):
    """Decode bytes that must cross HBM once per step: INT4 token-heads
    (codes + metadata), INT8 token-heads (codes + scale), block-table entries,
    the query and the bf16 output.  Append bytes: bf16 K/V read plus the INT4
    and (for protected positions) INT8 entries written."""
    d = w.d_h
    int4_th = 2 * (d // 2 + 4 * (d // w.group))   # K and V: codes + (Delta, m) per group
    int8_th = 2 * (d + 2)                         # K and V: codes + fp16 scale
    dec = 0
    n4_tok = 0
    n8_tok = 0
    for L in lens:
        L = int(L)
        n_p = min(L, w.sink + w.recent)
        n_4 = L - n_p
        n4_tok += n_4
        n8_tok += n_p
        dec += w.h_kv * (n_p * int8_th + n_4 * int4_th) + ((L + 15) // 16) * 4
    dec += len(lens) * w.h_q * d * 2 * 2            # q read + out write (bf16)
    app = len(lens) * w.h_kv * (2 * d * 2 + int4_th + int8_th) + len(lens) * 4 * 3
    return dec, app, n4_tok, n8_tok


class ClockSampler:
    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------- replicas (N > 1)

def reduce_max_ms(total_ms: float, world: int, device) -> float:
    """The slowest rank's timed-region length: every rank contributes its own
    CUDA-event time and all receive the maximum (NCCL on GPUs, gloo in
    the CPU tests).  A barrier precedes and follows the timed region."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(world: int, tokens_per_replica: int, ms_per_step: float) -> float:
    """Whole-job throughput of N independent replicas (weak scaling): every
    rank decodes its own copy of the workload in each step."""
    return world * tokens_per_replica / (ms_per_step / 1e3)


# --------------------------------------------------------------- workload

def run_step(cache, s, max_splits=0, ev=None):
    # (the KV4 cache only: a bf16 comparator cache, where built, is not part of the step)
    cache.append(s["k"], s["v"], s["seq"], s["pos"], s["lens"], comparator=False)
    if ev is not None:
        ev.record()
    cache.decode(s["q"], s["lens"], s["out"], s["lse"], max_splits=max_splits)


# ---------------------------------------------------------------- arms

def run_kv4(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from int8_kv_cache_kv4_gb300 import kv4
    kv4.load(build_if_missing=True)
    kv4.kv4_set_decode_kernel({"auto": kv4.KV4_KERNEL_AUTO, "stream": kv4.KV4_KERNEL_STREAM,
                               "mma": kv4.KV4_KERNEL_MMA_SYNC,
                               "cuda": kv4.KV4_KERNEL_CUDA_CORE}[args.kernel])

    w = W.WORKLOADS[args.workload]
    cache, s, lens, w = build_workload(w, dev, with_bf16=not args.no_bf16)
    # A second layer of the same shape (its own seeded K/V, query, outlier
    # channels and block table): the timed steps alternate between the two, as
    # consecutive layers of a model do, so that no step finds the previous
    # step's pages in L2.
    cache2, s2, _, _ = build_workload(w, dev, lens=lens, seed=w.seed + SECOND_LAYER_SEED)
    layers = [(cache, s), (cache2, s2)]
    dec_bytes, app_bytes, n4_tok, n8_tok = algorithmic_bytes(lens, w)
    tokens = int(lens.sum())
    stream = torch.cuda.current_stream()

    def steps(n):
        for i in range(n):
            run_step(*layers[i % 2], args.max_splits)

    steps(max(args.warmup, 2))
    torch.cuda.synchronize()
    for c, _ in layers:
        c.clear_status()
    # The K timed steps are launched as one CUDA graph captured from the
    # steps' C-ABI calls (append, then decode, per step), so that host-side
    # argument marshalling and per-graph launch gaps stay out of the steps;
    # inside it each call's kernels are programmatic dependents of the kernels
    # before them.  --no-graph launches the same calls eagerly.
    run_timed = lambda: steps(args.steps)  # noqa: E731
    if not args.no_graph:
        g_steps = _graph(run_timed)
        g_steps.replay()  # (the first replay uploads the graph)
        torch.cuda.synchronize()
        run_timed = g_steps.replay

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # Keep the GPU busy while the host enqueues the timed steps, so that the
    # events bracket back-to-back device work rather than host submission
    # latency.  The sleep precedes t0 and is not timed.
    torch.cuda._sleep(int(2.1e6 * max(5.0, 0.2 * args.steps)))
    t0.record(stream)
    run_timed()
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = t0.elapsed_time(t1)
    status = cache.read_status() | cache2.read_status()

    # The decode call's duration (the roofline's kernel time): the mean over
    # back-to-back calls alternating between the two layers, as in the steps;
    # and, beside it, single calls each behind an untimed GPU sleep.
    dec_fns = [lambda c=c, t=t: c.decode(t["q"], t["lens"], t["out"], t["lse"],  # noqa: E731
                                         max_splits=args.max_splits) for c, t in layers]
    n_dec = max(2 * args.steps, 40)
    dec_avg = _chained(dec_fns, n_dec, graph=not args.no_graph)
    app_fn = lambda: cache.append(s["k"], s["v"], s["seq"], s["pos"], s["lens"], comparator=False)  # noqa: E731
    dec_one = dec_fns[0]
    if not args.no_graph:
        dec_one, app_fn = _graph(dec_one).replay, _graph(app_fn).replay
    dec_iso = _timed(dec_one, warm=args.warmup, samples=max(args.steps, 20))
    app_t = _timed(app_fn, warm=args.warmup, samples=max(args.steps, 20))

    ms_per_step = reduce_max_ms(total_ms, world, dev) / args.steps
    value = replica_value(world, tokens, ms_per_step)
    hbm_peak, peak_kind = peaks()
    achieved = dec_bytes / (dec_avg / 1e3) / 1e9
    ksrc = kernel_source_hash()
    traffic = TRAFFIC.get((ksrc, w.name)) if args.kernel in ("auto", "stream") and args.max_splits == 0 else None

    # BF16-KV comparator on the same pages / inputs (reported beside, not in the step)
    comparator = None
    if not args.no_bf16:
        out16 = torch.empty_like(s["out"])
        for _ in range(3):
            cache.decode_bf16(s["q"], s["lens"], out16, None, max_splits=args.max_splits)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            cache.decode_bf16(s["q"], s["lens"], out16, None, max_splits=args.max_splits)
        e1.record(stream)
        torch.cuda.synchronize()
        bf_ms = e0.elapsed_time(e1) / args.steps
        bf_bytes = sum(w.h_kv * int(L) * 2 * w.d_h * 2 for L in lens) + len(lens) * w.h_q * w.d_h * 4
        drift = (s["out"].float() - out16.float()).abs()
        comparator = {"kernel": "bf16-KV paged decode on the tensor cores (same pages and block table)",
                      "ms": bf_ms, "tokens_per_s": tokens / (bf_ms / 1e3),
                      "algorithmic_GBps": bf_bytes / (bf_ms / 1e3) / 1e9,
                      "frac_of_hbm": bf_bytes / (bf_ms / 1e3) / 1e9 / hbm_peak,
                      "kv4_decode_speedup": bf_ms / dec_avg,
                      "byte_ratio_bound": bf_bytes / dec_bytes,
                      "output_drift_vs_bf16": {"max_abs": float(drift.max()),
                                               "mean_abs": float(drift.mean())}}

    # end to end through the public API with host buffers
    e2e = run_e2e(layers, args, stream)

    # the second configuration the target is stated on: one 128k-token
    # sequence (8 long pairs, each spread over many CTAs), its decode call
    # timed and held against the same roofline
    long_rec = None
    if not args.no_long and w.name != "long_128k":
        long_rec = decode_record(W.WORKLOADS["long_128k"], dev, args, hbm_peak, ksrc)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u4/i8 codes, f32 accumulate",
        "data": "synthetic (seeded N(0,1) bf16 K/V/q, outlier key channels x8)",
        "config": {"workload": w.name, "batch": int(len(lens)), "mean_len": float(lens.mean()),
                   "total_tokens": tokens, "h_q": w.h_q, "h_kv": w.h_kv, "d_h": w.d_h,
                   "sink": w.sink, "recent": w.recent, "group": w.group, "page": 16,
                   "splits": kv4.num_splits(cache.layout, int(len(lens)), args.max_splits),
                   "parallelism": f"replicas x{world}", "decode_kernel": args.kernel,
                   "layers": "steps alternate between two layer caches of this shape",
                   "launch": ("eager C-ABI calls" if args.no_graph else
                              "one CUDA graph of the K timed steps' C-ABI calls"),
                   "l2": "cache working set > L2, each step on the other layer (no flush needed)"},
        "decode_ms": dec_avg, "decode_ms_isolated": dec_iso["mean_ms"],
        "append_ms": app_t["mean_ms"],
        "append_exposed_ms": ms_per_step - dec_avg,
        "decode_tokens_per_s": tokens / (dec_avg / 1e3),
        "decode_algorithmic_GBps": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "kernel": decode_kernel_name(args, w),
                     "timed": (f"kv4_decode_attn calls (prep + decode kernels): CUDA events on "
                               f"the launching stream around {n_dec} back-to-back calls "
                               f"alternating two layers' caches, mean per call"),
                     "bytes_per_launch": dec_bytes, "peak_source": peak_kind,
                     "kernel_source_hash": ksrc},
        "append_algorithmic_bytes": app_bytes,
        # per step: quant_append_kernel, then the decode call's kernels
        # (stream_prep_kernel + decode_stream_kernel, and stream_merge_kernel
        # for few long pairs)
        "gpu_launches": (3 + (1 if _defers(w, len(lens)) else 0)) * args.steps,
        "clocks": clk,
        "device_status": status,
        "e2e": e2e,
        "bf16_comparator": comparator,
        "long_128k": long_rec,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, lens, budget_s=args.cpu_budget)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def decode_record(w: W.Workload, dev, args, hbm_peak, ksrc):
    """Decode call alone on workload w (two layer caches built and appended
    here): the mean per call over back-to-back calls alternating between the
    layers, the single-call time beside it, its algorithmic bytes and roofline
    fraction, and the kernel's DRAM traffic when a capture of these sources
    exists."""
    import torch
    cache, s, lens, w = build_workload(w, dev, with_bf16=False)
    cache2, s2, _, _ = build_workload(w, dev, lens=lens, seed=w.seed + SECOND_LAYER_SEED)
    layers = [(cache, s), (cache2, s2)]
    for c, t in layers:
        c.append(t["k"], t["v"], t["seq"], t["pos"], t["lens"])
        c.clear_status()
    dec_bytes, _, _, _ = algorithmic_bytes(lens, w)
    fns = [lambda c=c, t=t: c.decode(t["q"], t["lens"], t["out"], t["lse"],  # noqa: E731
                                     max_splits=args.max_splits) for c, t in layers]
    n = max(2 * args.steps, 40)
    ms = _chained(fns, n, graph=not args.no_graph)
    one = _graph(fns[0]).replay if not args.no_graph else fns[0]
    iso = _timed(one, warm=args.warmup, samples=max(args.steps, 20))
    achieved = dec_bytes / (ms / 1e3) / 1e9
    traffic = TRAFFIC.get((ksrc, w.name)) if args.kernel in ("auto", "stream") and args.max_splits == 0 else None
    rec = {"workload": w.name, "batch": int(len(lens)), "total_tokens": int(lens.sum()),
           "decode_ms": ms, "decode_ms_isolated": iso["mean_ms"],
           "decode_tokens_per_s": int(lens.sum()) / (ms / 1e3),
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                        "frac": achieved / hbm_peak, "traffic": traffic,
                        "kernel": decode_kernel_name(args, w), "bytes_per_launch": dec_bytes,
                        "timed": f"{n} back-to-back calls alternating two layers' caches"},
           "device_status": cache.read_status() | cache2.read_status()}
    del cache, s, cache2, s2, layers, fns, one
    torch.cuda.empty_cache()
    return rec


def _defers(w: W.Workload, num_seqs: int) -> bool:
    """Does the work-balanced decode merge its pairs in a separate kernel
    (few pairs, each spread over many CTAs: 8 pairs per CTA of the grid)?"""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return 8 * num_seqs * w.h_kv < 4 * sms  # (the grid: 4 CTAs per SM)


def decode_kernel_name(args, w):
    if args.kernel == "cuda" or w.d_h != 128 or w.h_q != 4 * w.h_kv:
        return "decode_split_kernel (CUDA cores, fused eq. A1 merge)"
    if args.kernel == "mma" or args.max_splits > 0:
        return "decode_mma_kernel (mma.sync split kernel, fused eq. A1 merge)"
    return "decode_stream_kernel (work-balanced, mma.sync, fused eq. A1 merge)"


def run_e2e(layers, args, stream):
    """The step through the binding with pinned host buffers, alternating the
    two layers like the timed steps: each step copies its new K/V token and
    query host -> device (one pinned buffer per layer, one copy), runs append +
    decode, and copies the output back.  Pipelined: the copies run on their own
    streams, so step i's input copy and step i-1's output copy overlap the
    kernels of the step before; events keep each layer's buffers from being
    rewritten before they are used.  Host clock around K steps.  The same steps
    run one after another (copy, kernels, copy) give `serial_ms_per_step`."""
    import torch
    dev = layers[0][1]["k"].device
    bufs = []
    for cache, s in layers:
        parts = [s["k"], s["v"], s["q"]]
        sizes = [t.numel() for t in parts]
        host = torch.empty(sum(sizes), dtype=torch.bfloat16).pin_memory()
        dev_in = torch.empty(sum(sizes), dtype=torch.bfloat16, device=dev)
        views, off = [], 0
        for t, n in zip(parts, sizes):
            host[off:off + n].copy_(t.reshape(-1).cpu())
            views.append(dev_in[off:off + n].view(t.shape))
            off += n
        hout = torch.empty(s["out"].shape, dtype=torch.bfloat16).pin_memory()
        bufs.append({"cache": cache, "s": dict(s, k=views[0], v=views[1], q=views[2]),
                     "host": host, "dev_in": dev_in, "hout": hout,
                     "h2d": torch.cuda.Event(), "done": torch.cuda.Event(),
                     "d2h": torch.cuda.Event()})
    h2d_stream, d2h_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def serial(i):
        b = bufs[i % 2]
        b["dev_in"].copy_(b["host"], non_blocking=True)
        run_step(b["cache"], b["s"], args.max_splits)
        b["hout"].copy_(b["s"]["out"], non_blocking=True)

    def pipelined(i):
        b = bufs[i % 2]
        with torch.cuda.stream(h2d_stream):
            h2d_stream.wait_event(b["done"])  # the layer's previous step has read its inputs
            b["dev_in"].copy_(b["host"], non_blocking=True)
            b["h2d"].record(h2d_stream)
        stream.wait_event(b["h2d"])
        stream.wait_event(b["d2h"])  # the layer's previous output has been copied out
        run_step(b["cache"], b["s"], args.max_splits)
        b["done"].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(b["done"])
            b["hout"].copy_(b["s"]["out"], non_blocking=True)
            b["d2h"].record(d2h_stream)

    def timed(fn):
        for i in range(4):
            fn(i)
        torch.cuda.synchronize()
        t = time.perf_counter()
        for i in range(args.steps):
            fn(i)
        torch.cuda.synchronize()
        return (time.perf_counter() - t) / args.steps

    dt_serial = timed(serial)
    dt = timed(pipelined)
    tokens = int(layers[0][1]["lens"].sum().item())
    return {"value": tokens / dt, "unit": UNIT, "h2d_bytes_per_step": bufs[0]["host"].numel() * 2,
            "d2h_bytes_per_step": bufs[0]["hout"].numel() * 2, "ms_per_step": dt * 1e3,
            "serial_ms_per_step": dt_serial * 1e3,
            "timed": "host clock around K steps through the binding, copies on their own streams"}


def _oracle_sources(w: W.Workload, lens, seqs):
    """Seeded host-side sources of the given sequences (numpy generator keyed
    by (seed, sequence), the recipe workloads.kv_numpy_block states)."""
    outl = W.outlier_channels(w.seed, w.h_kv, w.d_h)
    return {b: W.kv_numpy_block(w.seed, b, w.h_kv, int(lens[b]), w.d_h, outl) for b in seqs}


def _oracle_run(w: W.Workload, srcs, threads):
    """Quantize + fp64 decode of every sequence in srcs (all heads) on
    `threads` host threads.  The oracle is C behind ctypes, which releases
    the GIL for each call, so threads run sequences in parallel.  Returns the
    wall time in seconds."""
    import concurrent.futures as cf
    import oracle
    q = W.q_numpy(w.seed, 1, w.h_q, w.d_h)[0]
    kw = dict(g=w.group, S=w.sink, R=w.recent, sm_scale=1 / math.sqrt(w.d_h))
    t = time.perf_counter()
    if threads == 1:
        for k, v in srcs.values():
            oracle.decode_seq(q, k, v, **kw)
    else:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda kv: oracle.decode_seq(q, kv[0], kv[1], **kw), srcs.values()))
    return time.perf_counter() - t


def cpu_baseline(w: W.Workload, lens, budget_s=20.0, kind="oracle"):
    """The CPU oracle, as it stands, on a bounded sample of the workload
    (whole sequences, all heads): first on one host thread, then on every
    host core (one thread per core over sequences).  `value` is the all-cores
    throughput; both are reported with the sample they ran on."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    order = list(range(len(lens)))
    # one thread: consecutive sequences until half the budget is spent
    spent1, tok1, n1 = 0.0, 0, 0
    for b in order:
        spent1 += _oracle_run(w, _oracle_sources(w, lens, [b]), 1)
        tok1 += int(lens[b])
        n1 += 1
        if spent1 >= budget_s / 2:
            break
    rate1 = tok1 / spent1
    # all cores: as many whole sequences as the 1-thread rate says fill the
    # other half of the budget on every core (at least one per core)
    want = rate1 * (budget_s / 2) * cores
    seqs, tok = [], 0
    for b in order:
        if tok >= want and len(seqs) >= min(cores, len(order)):
            break
        seqs.append(b)
        tok += int(lens[b])
    srcs = _oracle_sources(w, lens, seqs)
    spent = _oracle_run(w, srcs, cores)
    return {"value": tok / spent, "unit": UNIT, "cores": cores, "kind": kind,
            "sample": f"{len(seqs)} of {len(lens)} sequences ({tok} tokens, all heads): quantize + "
                      f"fp64 decode on {cores} host threads in {spent:.2f} s",
            "one_thread": {"value": rate1, "unit": UNIT, "cores": 1,
                           "sample": f"{n1} sequences ({tok1} tokens, all heads) in {spent1:.2f} s"}}


def run_reference(args):
    """Reference arm: the CPU oracle as it stands on the machine's host cores.  A
    step is the quantize + fp64 decode of a fixed sample of the workload's
    sequences (all heads), sized from a short calibration so that all steps
    together take about --cpu-budget seconds; `ms_per_step` is the time a
    step actually took and `value` the tokens it processed per second."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = W.WORKLOADS[args.workload]
    lens = W.seq_lengths(w)
    cores = os.cpu_count() or 1
    # calibration (untimed): one thread on the shortest sequence
    b0 = int(np.argmin(lens))
    rate1 = int(lens[b0]) / _oracle_run(w, _oracle_sources(w, lens, [b0]), 1)
    per_step_s = max(0.5, args.cpu_budget / max(1, args.steps + args.warmup))
    want = rate1 * cores * per_step_s
    seqs, tok = [], 0
    for b in range(len(lens)):
        if tok >= want and len(seqs) >= min(cores, len(lens)):
            break
        seqs.append(b)
        tok += int(lens[b])
    srcs = _oracle_sources(w, lens, seqs)
    for _ in range(args.warmup):
        _oracle_run(w, srcs, cores)
    times = [_oracle_run(w, srcs, cores) for _ in range(args.steps)]
    ms = 1e3 * statistics.mean(times)
    value = tok / (ms / 1e3)
    sample = (f"each step: {len(seqs)} of {len(lens)} sequences ({tok} tokens, all heads), "
              f"quantize + fp64 decode on {cores} host threads; {sum(times):.1f} s timed")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "batch": int(len(lens)), "mean_len": float(lens.mean()),
                       "reference_step": f"{len(seqs)} sequences, {tok} tokens"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- report mode

def _timed(fn, warm=10, samples=90, flush=None):
    """CUDA-event times (ms) of fn on the current stream: `warm` untimed calls,
    then `samples` timed ones, each after an optional L2 flush."""
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(samples):
        if flush is not None:
            flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(210000)  # ~0.1 ms of untimed GPU work while the host enqueues e0, fn, e1
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    return {"median_ms": statistics.median(ts), "mean_ms": statistics.mean(ts)}


def _chained(fns, n, graph=True, reps=5):
    """Mean time (ms) per call of n back-to-back calls cycling through fns,
    CUDA events on the current stream around the whole chain (captured as one
    CUDA graph unless graph is False; median over reps chains, each behind an
    untimed GPU sleep)."""
    import torch

    def chain():
        for i in range(n):
            fns[i % len(fns)]()

    run = _graph(chain).replay if graph else chain
    run()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(int(2.1e6 * 3))  # ~3 ms of untimed GPU work while the host enqueues
        e0.record()
        run()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) / n)
    return statistics.median(ts)


def _graph(fn):
    """fn (one or more C-ABI calls) captured as a CUDA graph after one eager
    call (which also performs the library's one-time per-device setup)."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def run_report(args):
    """One JSON object per config of the pages' workloads (see workloads.py):
    decode time (median and mean of 90 CUDA-event samples after 10 warm-ups),
    resident KV tokens/s, algorithmic GB/s and its fraction of the measured HBM
    copy bandwidth, append time, the bf16-KV comparator, and the config's own
    variants.  Not the bench line: a per-configuration table."""
    import dataclasses
    import torch
    from int8_kv_cache_kv4_gb300 import kv4
    kv4.load(build_if_missing=True)
    dev = torch.device("cuda")
    hbm, peak_kind = peaks()
    l2_flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def decode_line(name, w, cache, s, lens, flush=False, extra=None):
        dec_b, app_b, _, _ = algorithmic_bytes(lens, w)
        f = (lambda: l2_flush.zero_()) if flush else None
        gd, ga = _graph(lambda: cache.decode(s["q"], s["lens"], s["out"], s["lse"])), \
            _graph(lambda: cache.append(s["k"], s["v"], s["seq"], s["pos"], s["lens"], comparator=False))
        td = _timed(gd.replay, flush=f)
        ta = _timed(ga.replay, flush=f)
        tok = int(lens.sum())
        line = {"report": name, "workload": w.name, "batch": int(len(lens)), "tokens": tok,
                "sink": w.sink, "recent": w.recent, "group": w.group,
                "decode": td, "append": ta, "decode_bytes": dec_b,
                "tokens_per_s": tok / (td["median_ms"] / 1e3),
                "GBps": dec_b / (td["median_ms"] / 1e3) / 1e9,
                "frac_of_hbm": dec_b / (td["median_ms"] / 1e3) / 1e9 / hbm, "peak": peak_kind,
                "l2_flushed": flush, "status": cache.read_status()}
        if extra:
            line.update(extra)
        print(json.dumps(line), flush=True)
        return line

    def bf16_line(name, w, cache, s, lens):
        out16 = torch.empty_like(s["out"])
        t = _timed(_graph(lambda: cache.decode_bf16(s["q"], s["lens"], out16, None)).replay)
        cache.decode(s["q"], s["lens"], s["out"], s["lse"])
        drift = (s["out"].float() - out16.float()).abs()
        b = sum(w.h_kv * int(L) * 2 * w.d_h * 2 for L in lens) + len(lens) * w.h_q * w.d_h * 4
        print(json.dumps({"report": name, "workload": w.name, "kernel": "bf16-KV decode", "decode": t,
                          "GBps": b / (t["median_ms"] / 1e3) / 1e9, "bytes": b,
                          "drift_vs_kv4": {"max_abs": float(drift.max()),
                                           "mean_abs": float(drift.mean())}}), flush=True)

    sel = set(args.report.split(",")) if args.report != "all" else {"1", "2", "3", "4", "5", "h", "c", "i8", "f4"}
    if "1" in sel:  # tiny: L2-resident, flushed
        w = W.WORKLOADS["tiny_b4_l512"]
        cache, s, lens, w = build_workload(w, dev)
        decode_line("config 1", w, cache, s, lens, flush=True)
        del cache
    if "2" in sel:
        w = W.WORKLOADS["qwen3_8b_b64"]
        cache, s, lens, w = build_workload(w, dev, with_bf16=True)
        decode_line("config 2", w, cache, s, lens)
        bf16_line("config 2", w, cache, s, lens)
        del cache
    if "3" in sel:  # 100 rollout steps: fresh token per sequence, append then decode
        w = W.WORKLOADS["rollout_b256"]
        cache, s, lens, w = build_workload(w, dev, extra_tokens=w.steps)
        from int8_kv_cache_kv4_gb300.cache import step_inputs
        steps = [step_inputs(w, len(lens), i, dev) for i in range(w.steps)]
        seq = s["seq"]
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(w.steps)]
        torch.cuda.synchronize()
        for i, (k, v, q) in enumerate(steps):
            pos = torch.as_tensor((lens - 1 + i).astype(np.int32), device=dev)
            ln = torch.as_tensor((lens + i).astype(np.int32), device=dev)
            ev[i][0].record()
            cache.append(k, v, seq, pos, ln)
            ev[i][1].record()
            cache.decode(q, ln, s["out"], s["lse"])
            ev[i][2].record()
        torch.cuda.synchronize()
        app = [e[0].elapsed_time(e[1]) for e in ev]
        dec = [e[1].elapsed_time(e[2]) for e in ev]
        dec_b, _, _, _ = algorithmic_bytes(lens + w.steps // 2, w)
        print(json.dumps({"report": "config 3", "workload": w.name, "steps": w.steps,
                          "append_ms": {"median": statistics.median(app), "mean": statistics.mean(app)},
                          "decode_ms": {"median": statistics.median(dec), "mean": statistics.mean(dec)},
                          "step_ms_mean": statistics.mean(a + d for a, d in zip(app, dec)),
                          "decode_GBps_mid": dec_b / (statistics.median(dec) / 1e3) / 1e9,
                          "frac_of_hbm_mid": dec_b / (statistics.median(dec) / 1e3) / 1e9 / hbm,
                          "resident_tokens_mid": int((lens + w.steps // 2).sum()),
                          "status": cache.read_status()}), flush=True)
        del cache, steps
    if "4" in sel:  # long context: mixed, INT8 everywhere (R >= L), bf16
        w = W.WORKLOADS["long_128k"]
        cache, s, lens, w = build_workload(w, dev, with_bf16=True)
        decode_line("config 4 mixed", w, cache, s, lens)
        bf16_line("config 4", w, cache, s, lens)
        del cache
        w8 = dataclasses.replace(w, recent=int(lens.max()))
        cache, s, lens, w8 = build_workload(w8, dev)
        decode_line("config 4 int8 everywhere", w8, cache, s, lens)
        del cache
    if "f4" in sel:  # representation drift against bf16 attention: affine INT4 vs NVFP4 / MXFP4
        w = W.WORKLOADS["qwen3_8b_b64"]
        ref_cache, s, lens, w = build_workload(w, dev, with_bf16=True)
        ref = torch.empty_like(s["out"])
        ref_cache.append(s["k"], s["v"], s["seq"], s["pos"], s["lens"])
        ref_cache.decode_bf16(s["q"], s["lens"], ref, None)
        torch.cuda.synchronize()
        del ref_cache
        variants = [("affine INT4 g32 + INT8 S4 R128 (deployed)", dict()),
                    ("affine INT4 g128, no protection", dict(group=128, recent=0)),
                    ("affine INT4 g128, no protection, K rotated", dict(group=128, recent=0, hadamard_k=True)),
                    ("NVFP4", dict(fp4=kv4.KV4_FP4_NVFP4)),
                    ("NVFP4, K rotated", dict(fp4=kv4.KV4_FP4_NVFP4, hadamard_k=True)),
                    ("MXFP4", dict(fp4=kv4.KV4_FP4_MXFP4)),
                    ("MXFP4, K rotated", dict(fp4=kv4.KV4_FP4_MXFP4, hadamard_k=True))]
        for name, kw in variants:
            wv = w if "group" not in kw else dataclasses.replace(w, sink=0 if kw.get("recent") == 0 else w.sink)
            cache, s2, lens2, _ = build_workload(wv, dev, **kw)
            cache.append(s2["k"], s2["v"], s2["seq"], s2["pos"], s2["lens"])
            cache.decode(s2["q"], s2["lens"], s2["out"], s2["lse"])
            torch.cuda.synchronize()
            d = (s2["out"].float() - ref.float()).abs()
            print(json.dumps({"report": "representation drift vs bf16 attention", "workload": w.name,
                              "representation": name, "max_abs": float(d.max()),
                              "mean_abs": float(d.mean()), "status": cache.read_status()}), flush=True)
            del cache
            torch.cuda.empty_cache()
    if "i8" in sel:  # tensor-pipe rates behind the integer decode variant (libkv4_diag.so)
        from int8_kv_cache_kv4_gb300 import diag
        sink = torch.zeros(1, dtype=torch.int32, device=dev)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        for kind, name, blocks, iters in (
                (diag.KIND_MMA_F16, "mma.sync m16n8k16 fp16 (fp32 accumulate)", sms * 8, 4096),
                (diag.KIND_MMA_I8, "mma.sync m16n8k32 int8 (int32 accumulate)", sms * 8, 4096),
                (diag.KIND_TC_F16, "tcgen05.mma kind::f16 128x256x16 (fp32 in tensor memory)",
                 sms, 4096)):
            t = _timed(lambda: diag.kv4_diag_mma_rate(kind, blocks, iters, sink), warm=3, samples=10)
            print(json.dumps({"report": "mma rate", "kind": name, "ms": t["median_ms"],
                              "TOPS": diag.ops(kind, blocks, iters) / (t["median_ms"] / 1e3) / 1e12,
                              "status": int(sink.item())}), flush=True)
        print(json.dumps({"report": "mma rate", "kind": "tcgen05.mma kind::i8",
                          "unavailable": "ptxas rejects it for sm_103a"}), flush=True)
    if "c" in sel:  # KV concentration: continuous refill vs synchronous waves, driven on the GPU
        from int8_kv_cache_kv4_gb300 import rollout as RO
        w = W.WORKLOADS["rollout_b256"]
        sup, pmf = W.lognormal_length_pmf(w.length, w.sigma, w.length_lo, w.length_hi)
        shape = dict(h_q=w.h_q, h_kv=w.h_kv, d_h=w.d_h, group=w.group, sink=w.sink,
                     recent=w.recent)
        waves = RO.wave_schedule(w.batch, args.prompt, sup, pmf, args.waves,
                                 np.random.default_rng([w.seed, 30]))
        refill = RO.refill_schedule(w.batch, args.prompt, sup, pmf, waves.steps,
                                    np.random.default_rng([w.seed, 31]))
        lines = {}
        for sched in (refill, waves):
            res = RO.drive(sched, seed=w.seed, **shape)
            lines[sched.kind] = RO.report(sched, res, **shape)
            del res
            torch.cuda.empty_cache()
            print(json.dumps(dict({"report": "config 3 concentration", "workload": w.name,
                                   "lengths": "lognormal(median 3000, sigma 0.8) clipped to [256, 16384]",
                                   "peak_GBps": hbm}, **lines[sched.kind])), flush=True)
        r, wv = lines["refill"], lines["waves"]
        print(json.dumps({"report": "config 3 concentration ratio",
                          "volume_ratio_measured": r["volume_tokens"] / wv["volume_tokens"],
                          "decode_ms_ratio": r["decode_ms_mean"] / wv["decode_ms_mean"],
                          "occupancy_waves": wv["active"], "steps_each": waves.steps}), flush=True)
    if "h" in sel:  # Hadamard K-rotation on the batch-64 layer: rotated append, query rotation
        w = W.WORKLOADS["qwen3_8b_b64"]
        cache, s, lens, w = build_workload(w, dev, hadamard_k=True)
        q_rot = torch.empty_like(s["q"])
        tq = _timed(_graph(lambda: kv4.kv4_hadamard_bf16(s["q"], q_rot)).replay)
        qb = 2 * s["q"].numel() * 2
        # decode here includes the query rotation (MixedKVCache.decode rotates q)
        decode_line("config 2 hadamard-k", w, cache, s, lens,
                    extra={"query_rotation": tq,
                           "query_rotation_GBps": qb / (tq["median_ms"] / 1e3) / 1e9})
        del cache
    if "5" in sel:  # the 36-layer step: every layer appended and decoded, one graph per step
        w = W.WORKLOADS["qwen3_8b_36l"]
        base = {}
        for g in (32, 64, 128):
            for R in (0, 64, 128, 512):
                layers = []
                for layer in range(w.layers):  # independent seeds 500 + layer
                    cache, s, lens, wl = build_workload(w, dev, group=g, recent=R,
                                                        seed=w.seed + layer)
                    layers.append((cache, s))
                dec_b, app_b, _, _ = algorithmic_bytes(lens, wl)

                def step():
                    for cache, s in layers:
                        cache.append(s["k"], s["v"], s["seq"], s["pos"], s["lens"])
                        cache.decode(s["q"], s["lens"], s["out"], s["lse"])

                def decodes():
                    for cache, s in layers:
                        cache.decode(s["q"], s["lens"], s["out"], s["lse"])

                t_step = _timed(_graph(step).replay, warm=3, samples=10)
                t_dec = _timed(_graph(decodes).replay, warm=3, samples=10)
                st = [c.read_status() for c, _ in layers]
                tok = int(lens.sum())
                if R == 0:
                    base[g] = t_step["median_ms"]
                print(json.dumps({
                    "report": "config 5: 36-layer step", "workload": w.name, "group": g,
                    "recent": R, "layers": w.layers, "batch": int(len(lens)),
                    "tokens_per_layer": tok,
                    "step_ms": t_step, "decode_only_ms": t_dec,
                    "decode_ms_per_layer": t_dec["median_ms"] / w.layers,
                    "decode_bytes_per_layer": dec_b,
                    "decode_GBps": dec_b * w.layers / (t_dec["median_ms"] / 1e3) / 1e9,
                    "decode_frac_of_hbm": dec_b * w.layers / (t_dec["median_ms"] / 1e3) / 1e9 / hbm,
                    "tokens_per_s_per_layer": tok * w.layers / (t_step["median_ms"] / 1e3),
                    "step_cost_vs_R0": t_step["median_ms"] / base[g],
                    "status": max(st)}), flush=True)
                del layers, cache, s
                torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kv4", choices=["kv4", "reference"])
    ap.add_argument("--workload", default="qwen3_8b_b64", choices=sorted(W.WORKLOADS))
    ap.add_argument("--max-splits", type=int, default=0)
    ap.add_argument("--kernel", default="auto", choices=["auto", "stream", "mma", "cuda"],
                    help="decode kernel (auto = the fastest measured for the layout)")
    ap.add_argument("--no-long", action="store_true",
                    help="skip the long_128k decode record beside the step")
    ap.add_argument("--no-bf16", action="store_true", help="skip the bf16-KV comparator")
    ap.add_argument("--no-graph", action="store_true", help="time eager calls, not graph replays")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time")
    ap.add_argument("--waves", type=int, default=2,
                    help="synchronous waves of the driven rollout schedules (--report c)")
    ap.add_argument("--prompt", type=int, default=256,
                    help="prompt length P of the driven rollout schedules (--report c)")
    ap.add_argument("--report", default=None,
                    help="instead of the bench line: per-config report for configs 'all' or e.g. '2,4'")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.report:
        run_report(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_kv4(args)


if __name__ == "__main__":
    main()
