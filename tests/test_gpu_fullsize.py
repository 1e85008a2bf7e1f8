"""Full-size parity: the workloads at their stated sizes, run through the C ABI
in the launch configuration the benchmark times, checked against the CPU
oracle on a seeded sample of sequences (all heads): the cache bytes of every
position of a sampled sequence bit for bit, and the decode outputs within the
tolerance.  Sequence sources are regenerated from their seeds."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

import oracle  # noqa: E402
from kv4_case import compare_outputs, oracle_decode_many  # noqa: E402
from int8_kv_cache_kv4_gb300 import kv4, workloads as W  # noqa: E402
from int8_kv_cache_kv4_gb300.cache import build_workload, source_kv, step_inputs  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kv4.load(build_if_missing=True)


def _check_seq_bytes(cache, w, b, k_src, v_src, L, rotate_k=False):
    """Oracle-append sequence b's L positions into a private pool (page p at
    pool page p) and compare every page chunk and the side block with the
    device cache."""
    npages = (L + 15) // 16
    cb = oracle.chunk_bytes(w.d_h, w.group)
    sb = oracle.side_block_bytes(w.d_h, w.sink, w.recent)
    paged = np.zeros(npages * w.h_kv * cb, np.uint8)
    side = np.zeros(max(16, w.h_kv * sb), np.uint8)
    bt = np.arange(npages, dtype=np.int32)[None, :]
    st = oracle.quant_append(h_kv=w.h_kv, d_h=w.d_h, g=w.group, S=w.sink, R=w.recent, max_seqs=1,
                             num_pages=npages, max_pages_per_seq=npages, paged=paged, side=side,
                             k_new=np.ascontiguousarray(k_src.transpose(1, 0, 2)),
                             v_new=np.ascontiguousarray(v_src.transpose(1, 0, 2)),
                             tok_seq=np.zeros(L, np.int32), tok_pos=np.arange(L, dtype=np.int32),
                             seq_lens=np.array([L], np.int32), block_table=bt, rotate_k=rotate_k)
    assert st == 0
    dev_bt = cache.block_table[b, :npages].cpu().numpy()
    allp = cache.paged.view(-1, w.h_kv * cb)
    got = allp[torch.as_tensor(dev_bt.astype(np.int64), device=allp.device)].cpu().numpy().ravel()
    assert np.array_equal(got, paged), f"seq {b}: INT4 page bytes differ from the oracle"
    if w.sink + w.recent > 0:
        gs = cache.side[b * w.h_kv * sb:(b + 1) * w.h_kv * sb].cpu().numpy()
        assert np.array_equal(gs, side[: w.h_kv * sb]), f"seq {b}: side cache differs"


def _check_decode(out, lse, w, seqs, srcs, qs, lens, rotate_k=False):
    """Decode outputs of the sampled sequences against the oracle (run on the
    host's cores), with the raw statistics of compare_outputs."""
    kw = dict(g=w.group, S=w.sink, R=w.recent, sm_scale=1 / math.sqrt(w.d_h), rotate_k=rotate_k)
    jobs = {b: (oracle.hadamard_bf16(qs[b]) if rotate_k else qs[b], srcs[b][0], srcs[b][1], kw)
            for b in seqs}
    ref_o, ref_l = oracle_decode_many(jobs)
    return compare_outputs(out, lse, ref_o, ref_l, seqs, lens,
                           label=f"{w.name} g={w.group} R={w.recent} ({len(seqs)} seqs):")


def _run_step(cache, s):
    cache.append(s["k"], s["v"], s["seq"], s["pos"], s["lens"])
    cache.decode(s["q"], s["lens"], s["out"], s["lse"])
    torch.cuda.synchronize()
    assert cache.read_status() == 0
    return (s["out"].float().cpu().numpy().astype(np.float64),
            s["lse"].cpu().numpy().astype(np.float64))


def _sample(w, lens, n=8):
    return W.sample_rows(w.seed, len(lens), n, extra=[int(np.argmin(lens)), int(np.argmax(lens))])


def test_qwen3_8b_batch64_full_size():
    # every one of the 64 sequences' outputs; the cache bytes of 8 + 2 sequences
    w = W.WORKLOADS["qwen3_8b_b64"]
    dev = torch.device("cuda")
    cache, s, lens, w = build_workload(w, dev)
    out, lse = _run_step(cache, s)
    qs = s["q"].view(torch.int16).cpu().numpy().view(np.uint16)
    seqs = list(range(len(lens)))
    srcs = {b: source_kv(w, b, int(lens[b]), dev) for b in seqs}
    for b in _sample(w, lens, 8):
        _check_seq_bytes(cache, w, b, *srcs[b], int(lens[b]))
    # (outputs reach |o| = 2.2 here, where one bf16 ulp is 2^-6: the element
    # rule of compare_outputs applies; the raw mean meets 2e-4 as it stands)
    _, mean = _check_decode(out, lse, w, seqs, srcs, qs, lens)
    assert mean <= 2e-4


def test_qwen3_8b_batch64_full_size_hadamard_k():
    # the same layer with the K rotation on append and the query rotation
    w = W.WORKLOADS["qwen3_8b_b64"]
    dev = torch.device("cuda")
    cache, s, lens, w = build_workload(w, dev, hadamard_k=True)
    out, lse = _run_step(cache, s)
    seqs = _sample(w, lens, 8)
    qs = s["q"].view(torch.int16).cpu().numpy().view(np.uint16)
    srcs = {b: source_kv(w, b, int(lens[b]), dev) for b in seqs}
    for b in seqs[:8]:
        _check_seq_bytes(cache, w, b, *srcs[b], int(lens[b]), rotate_k=True)
    _, mean = _check_decode(out, lse, w, seqs, srcs, qs, lens, rotate_k=True)
    assert mean <= 2e-4


@pytest.mark.parametrize("recent", [256, 131072])
def test_long_context_128k(recent):
    # mixed INT4/INT8 (R = 256) and INT8-everywhere (R >= L, same code path)
    w = W.WORKLOADS["long_128k"]
    dev = torch.device("cuda")
    cache, s, lens, w = build_workload(w, dev, recent=recent)
    out, lse = _run_step(cache, s)
    qs = s["q"].view(torch.int16).cpu().numpy().view(np.uint16)
    srcs = {0: source_kv(w, 0, int(lens[0]), dev)}
    _check_seq_bytes(cache, w, 0, *srcs[0], int(lens[0]))
    mx, mean = _check_decode(out, lse, w, [0], srcs, qs, lens)
    assert mx <= 2e-3 and mean <= 2e-4


def test_rollout_batch256_100_steps():
    """100 append + decode steps over 256 sequences.  Checked: every appended
    token's INT4 codes and metadata (all 256 x 100 tokens, all heads) and its
    INT8 side entry (every appended position is still inside the final recent
    window: 100 < R), bit for bit; the final decode on 8 + 2 sampled sequences
    with their whole history."""
    w = W.WORKLOADS["rollout_b256"]
    dev = torch.device("cuda")
    steps = w.steps
    assert steps < w.recent
    cache, s, lens0, w = build_workload(w, dev, extra_tokens=steps)
    B = len(lens0)
    _run_step(cache, s)
    ks, vs = [s["k"].view(torch.int16).cpu().numpy().view(np.uint16)], \
        [s["v"].view(torch.int16).cpu().numpy().view(np.uint16)]
    for st in range(1, steps):
        k, v, q = step_inputs(w, B, st, dev)
        ks.append(k.view(torch.int16).cpu().numpy().view(np.uint16))
        vs.append(v.view(torch.int16).cpu().numpy().view(np.uint16))
        lens = lens0 + st
        s2 = dict(s, k=k, v=v, q=q, pos=torch.as_tensor((lens - 1).astype(np.int32), device=dev),
                  lens=torch.as_tensor(lens.astype(np.int32), device=dev))
        out, lse = _run_step(cache, s2)
    lens = lens0 + steps - 1
    # --- every appended token: oracle bytes in a private pool (pages of each
    # sequence's appended span only) against the device slots
    first = (lens0 - 1) // 16
    npg = (lens0 - 1 + steps - 1) // 16 - first + 1
    off = np.concatenate([[0], np.cumsum(npg)])
    mpps = int(cache.block_table.shape[1])
    bt_priv = np.zeros((B, mpps), np.int32)
    for b in range(B):
        bt_priv[b, first[b]:first[b] + npg[b]] = off[b] + np.arange(npg[b])
    cb = oracle.chunk_bytes(w.d_h, w.group)
    sb = oracle.side_block_bytes(w.d_h, w.sink, w.recent)
    paged = np.zeros(int(off[-1]) * w.h_kv * cb, np.uint8)
    side = np.zeros(B * w.h_kv * sb, np.uint8)
    T = B * steps
    st = oracle.quant_append(h_kv=w.h_kv, d_h=w.d_h, g=w.group, S=w.sink, R=w.recent, max_seqs=B,
                             num_pages=int(off[-1]), max_pages_per_seq=mpps, paged=paged, side=side,
                             k_new=np.concatenate(ks), v_new=np.concatenate(vs),
                             tok_seq=np.tile(np.arange(B, dtype=np.int32), steps),
                             tok_pos=np.concatenate([(lens0 - 1 + i).astype(np.int32)
                                                     for i in range(steps)]),
                             seq_lens=lens.astype(np.int32), block_table=bt_priv)
    assert st == 0 and T == len(np.concatenate(ks))
    bt_dev = cache.block_table.cpu().numpy()
    pages_dev = np.unique(np.concatenate([bt_dev[b, first[b]:first[b] + npg[b]] for b in range(B)]))
    dev_pool = cache.paged.view(-1, w.h_kv * cb)
    got = dev_pool[torch.as_tensor(pages_dev.astype(np.int64), device=dev_pool.device)].cpu().numpy()
    where = {int(p): i for i, p in enumerate(pages_dev)}
    got = got.ravel()
    side_dev = cache.side.cpu().numpy()
    d, ng = w.d_h, w.d_h // w.group
    row, meta = d // 2, 4 * ng

    def rel(slot):
        """Byte offsets of one slot inside a chunk: its K row, V row, K meta
        and, per group, its V Delta and V m entries (quad (slot % 8) // 2,
        entry 2 (slot // 8) + slot % 2 of the quad)."""
        ent = np.array([((slot % 8) // 2 * ng + j) * 4 + 2 * (slot // 8) + slot % 2
                        for j in range(ng)])
        vmeta = np.concatenate([32 * row + 16 * meta + 2 * ent[:, None] + np.arange(2),
                                32 * row + 24 * meta + 2 * ent[:, None] + np.arange(2)]).ravel()
        return np.concatenate([slot * row + np.arange(row), 16 * row + slot * row + np.arange(row),
                               32 * row + slot * meta + np.arange(meta), vmeta])

    ns, nsp = w.sink + w.recent, oracle.side_scale_entries(w.sink, w.recent)

    def srel(ring):  # one side slot: K8 row, V8 row, K8 scale, V8 scale
        return np.concatenate([ring * d + np.arange(d), (ns + ring) * d + np.arange(d),
                               2 * ns * d + 2 * ring + np.arange(2),
                               2 * ns * d + 2 * nsp + 2 * ring + np.arange(2)])

    hs = np.arange(w.h_kv)
    bad = 0
    for i in range(steps):
        p = (lens0 - 1 + i).astype(np.int64)
        pd = np.array([where[int(bt_dev[b, p[b] // 16])] for b in range(B)], np.int64)
        pp = bt_priv[np.arange(B), p // 16].astype(np.int64)
        r_int4 = np.stack([rel(int(t)) for t in p % 16])                     # [B][160]
        i_dev = ((pd[:, None] * w.h_kv + hs[None, :]) * cb)[:, :, None] + r_int4[:, None, :]
        i_ora = ((pp[:, None] * w.h_kv + hs[None, :]) * cb)[:, :, None] + r_int4[:, None, :]
        bad += int((got[i_dev] != paged[i_ora]).any(axis=2).sum())
        r_side = np.stack([srel(int(w.sink + t % w.recent)) for t in p])      # [B][260]
        i_side = ((np.arange(B)[:, None] * w.h_kv + hs[None, :]) * sb)[:, :, None] + r_side[:, None, :]
        bad += int((side_dev[i_side] != side[i_side]).any(axis=2).sum())
    assert bad == 0, f"{bad} appended token-head entries differ from the oracle"
    # --- final decode over whole histories on a sample
    seqs = _sample(w, lens, 8)
    qs = q.view(torch.int16).cpu().numpy().view(np.uint16)
    srcs = {b: source_kv(w, b, int(lens0[b]), dev, steps=steps) for b in seqs}
    for b in seqs[:2]:
        _check_seq_bytes(cache, w, b, *srcs[b], int(lens[b]))
    _, mean = _check_decode(out, lse, w, seqs, srcs, qs, lens)
    assert mean <= 2e-4


def test_36_layer_workload_two_layers():
    # two independently seeded layers (seeds 500 and 501) of the 128 x 8192
    # step at its configured point (R = 128, group 32): every sampled
    # sequence's cache bytes and decode outputs, per layer
    w0 = W.WORKLOADS["qwen3_8b_36l"]
    dev = torch.device("cuda")
    for layer in (0, 1):
        cache, s, lens, w = build_workload(w0, dev, seed=w0.seed + layer)
        out, lse = _run_step(cache, s)
        seqs = W.sample_rows(w.seed, len(lens), 8)
        qs = s["q"].view(torch.int16).cpu().numpy().view(np.uint16)
        srcs = {b: source_kv(w, b, int(lens[b]), dev) for b in seqs}
        for b in seqs:
            _check_seq_bytes(cache, w, b, *srcs[b], int(lens[b]))
        _, mean = _check_decode(out, lse, w, seqs, srcs, qs, lens)
        assert mean <= 2e-4
        del cache
        torch.cuda.empty_cache()


@pytest.mark.parametrize("recent,group", [(0, 32), (128, 64), (512, 128), (64, 32)])
def test_36_layer_workload_one_layer(recent, group):
    # one layer (seed 500) of the 128 x 8192 step at points of the R x group sweep
    w = W.WORKLOADS["qwen3_8b_36l"]
    dev = torch.device("cuda")
    cache, s, lens, w = build_workload(w, dev, recent=recent, group=group)
    out, lse = _run_step(cache, s)
    seqs = _sample(w, lens, 8)
    qs = s["q"].view(torch.int16).cpu().numpy().view(np.uint16)
    srcs = {b: source_kv(w, b, int(lens[b]), dev) for b in seqs}
    for b in seqs[:8]:
        _check_seq_bytes(cache, w, b, *srcs[b], int(lens[b]))
    _, mean = _check_decode(out, lse, w, seqs, srcs, qs, lens)
    assert mean <= 2e-4
    del cache
    torch.cuda.empty_cache()
