"""Pins for the oracle's packed quantize-on-append (the expected cache bytes).

The byte layout is the library's documented one (16-token pages; per page and
kv head: K codes, V codes, K meta, V meta; low nibble = even channel; side
cache with S sink slots and an R-slot ring).  These tests parse the bytes
back by that description and tie them to the oracle's element encoders, the
protection rule of KV4-RL Sec. 5.2 and the "INT4 history covers every
position" rule of App. A.3.
"""
import numpy as np
import pytest

import oracle
from int8_kv_cache_kv4_gb300 import workloads as W

CANARY = 0xA5


def _unpack_chunk(chunk, d_h, g):
    """Parse one (page, kv head) chunk back into per-slot codes and (Delta, m)
    of K and V, following the layout description of include/kv4.h."""
    ng = d_h // g
    nb = d_h // 32
    kc = chunk[: 16 * d_h // 2].reshape(16, d_h // 2)
    vc = chunk[16 * d_h // 2: 16 * d_h].reshape(16, d_h // 2)
    kmeta = chunk[16 * d_h: 16 * d_h + 64 * ng].view(np.uint16).reshape(16, ng, 2)
    vd = chunk[16 * d_h + 64 * ng: 16 * d_h + 96 * ng].view(np.uint16).reshape(4, ng, 4)
    vm = chunk[16 * d_h + 96 * ng: 16 * d_h + 128 * ng].view(np.uint16).reshape(4, ng, 4)
    vmeta = np.empty((16, ng, 2), dtype=np.uint16)
    for t in range(16):       # quad t%8 // 2, entry 2 (t // 8) + t % 2 of the quad
        vmeta[t, :, 0] = vd[(t % 8) // 2, :, 2 * (t // 8) + t % 2]
        vmeta[t, :, 1] = vm[(t % 8) // 2, :, 2 * (t // 8) + t % 2]

    def nib(rows):
        out = np.empty((16, d_h), dtype=np.uint8)
        out[:, 0::2] = rows & 0xF
        out[:, 1::2] = rows >> 4
        return out

    # V rows: 16-byte piece P of slot t sits at piece position P ^ ((t >> 1) % npieces)
    def unswizzle_v(rows):
        out = np.empty_like(rows)
        for t in range(16):
            for P in range(nb):
                phys = P ^ ((t >> 1) % nb)
                out[t, 16 * P:16 * P + 16] = rows[t, 16 * phys:16 * phys + 16]
        return out

    # K rows: word b of quarter q (at word index nb q + b) holds channels 32 b + 8 q .. + 7
    def unpermute_k(rows):
        out = np.empty_like(rows)
        for q in range(4):
            for b in range(nb):
                w = nb * q + b
                c = 32 * b + 8 * q
                out[:, c // 2: c // 2 + 4] = rows[:, 4 * w: 4 * w + 4]
        return out
    return nib(unpermute_k(kc)), nib(unswizzle_v(vc)), kmeta, vmeta


def _unswizzle8(rows):
    """Undo the side cache's piece order: 16-byte piece P of slot t sits at
    piece position P ^ (t % (d_h / 16))."""
    n, d_h = rows.shape
    out = np.empty_like(rows)
    for t in range(n):
        for P in range(d_h // 16):
            src = P ^ (t % (d_h // 16))
            out[t, 16 * P:16 * P + 16] = rows[t, 16 * src:16 * src + 16]
    return out


def _side_block(side, s, h, h_kv, d_h, S, R):
    sb = oracle.side_block_bytes(d_h, S, R)
    NS = S + R
    blk = side[(s * h_kv + h) * sb:(s * h_kv + h + 1) * sb]
    k8 = _unswizzle8(blk[: NS * d_h].view(np.int8).reshape(NS, d_h))
    v8 = _unswizzle8(blk[NS * d_h: 2 * NS * d_h].view(np.int8).reshape(NS, d_h))
    NSP = (NS + 7) // 8 * 8  # scale arrays padded to a multiple of 8 entries
    ks = blk[2 * NS * d_h: 2 * NS * d_h + 2 * NS].view(np.uint16)
    vs = blk[2 * NS * d_h + 2 * NSP: 2 * NS * d_h + 2 * NSP + 2 * NS].view(np.uint16)
    return k8, v8, ks, vs


def _setup(h_kv=2, d_h=64, g=32, S=2, R=4, max_seqs=3, num_pages=12, mpps=4):
    paged = np.full(num_pages * h_kv * oracle.chunk_bytes(d_h, g), CANARY, dtype=np.uint8)
    side = np.full(max_seqs * h_kv * oracle.side_block_bytes(d_h, S, R), CANARY, dtype=np.uint8)
    return dict(h_kv=h_kv, d_h=d_h, g=g, S=S, R=R, max_seqs=max_seqs, num_pages=num_pages,
                max_pages_per_seq=mpps), paged, side


@pytest.mark.parametrize("g", [16, 32, 64])
def test_single_token_touches_only_its_slot(g):
    lay, paged, side = _setup(g=g)
    h_kv, d_h = lay["h_kv"], lay["d_h"]
    bt = np.full((3, 4), -1, dtype=np.int32)
    bt[1] = [7, 2, 9, 0]
    k, v = W.kv_numpy_block(1, 0, h_kv, 1, d_h, W.outlier_channels(1, h_kv, d_h))
    k = np.ascontiguousarray(k.transpose(1, 0, 2))
    v = np.ascontiguousarray(v.transpose(1, 0, 2))
    pos = 21                       # page index 1 -> physical page 2, slot 5
    lens = np.array([0, 30, 0], dtype=np.int32)
    before = paged.copy()
    st = oracle.quant_append(**lay, paged=paged, side=side, k_new=k, v_new=v,
                             tok_seq=np.array([1]), tok_pos=np.array([pos]), seq_lens=lens,
                             block_table=bt)
    assert st == 0
    cb = oracle.chunk_bytes(d_h, g)
    changed = np.nonzero(paged != before)[0]
    assert changed.min() >= 2 * h_kv * cb and changed.max() < 3 * h_kv * cb
    for h in range(h_kv):
        chunk = paged[(2 * h_kv + h) * cb:(2 * h_kv + h + 1) * cb]
        kc, vc, km, vm = _unpack_chunk(chunk, d_h, g)
        ck, dk, mk, _ = oracle.int4_encode(W.bf16_bits_to_f32(k[0, h]), g)
        cv, dv, mv, _ = oracle.int4_encode(W.bf16_bits_to_f32(v[0, h]), g)
        assert np.array_equal(kc[5], ck) and np.array_equal(vc[5], cv)
        assert np.array_equal(km[5, :, 0], dk) and np.array_equal(km[5, :, 1], mk)
        assert np.array_equal(vm[5, :, 0], dv) and np.array_equal(vm[5, :, 1], mv)
        # other slots untouched (still canary)
        raw = chunk.reshape(-1)
        assert np.all(raw[: 5 * d_h // 2] == CANARY)
    # position 21 of a 30-long sequence with S=2, R=4 is not protected
    assert np.all(side == CANARY)


def test_bulk_append_side_cache_holds_sinks_and_final_window():
    lay, paged, side = _setup(S=2, R=4)
    h_kv, d_h, S, R = lay["h_kv"], lay["d_h"], lay["S"], lay["R"]
    L = 27
    bt = np.full((3, 4), -1, dtype=np.int32)
    bt[2] = [3, 1, 11, -1]
    k, v = W.kv_numpy_block(2, 0, h_kv, L, d_h, W.outlier_channels(2, h_kv, d_h))
    kt = np.ascontiguousarray(k.transpose(1, 0, 2))
    vt = np.ascontiguousarray(v.transpose(1, 0, 2))
    # tokens in a scrambled order: the result must not depend on it
    order = np.random.default_rng(3).permutation(L)
    st = oracle.quant_append(**lay, paged=paged, side=side, k_new=kt[order], v_new=vt[order],
                             tok_seq=np.full(L, 2), tok_pos=order.astype(np.int32),
                             seq_lens=np.array([0, 0, L], dtype=np.int32), block_table=bt)
    assert st == 0
    for h in range(h_kv):
        k8, v8, ks, vs = _side_block(side, 2, h, h_kv, d_h, S, R)
        ck, sk, _ = oracle.int8_encode(W.bf16_bits_to_f32(k[h]))
        cv, sv, _ = oracle.int8_encode(W.bf16_bits_to_f32(v[h]))
        for p in [0, 1, 23, 24, 25, 26]:       # sinks and the last R = 4 positions
            slot = p if p < S else S + p % R
            assert np.array_equal(k8[slot], ck[p]) and ks[slot] == sk[p]
            assert np.array_equal(v8[slot], cv[p]) and vs[slot] == sv[p]
        # every position has its INT4 entry (App. A.3)
        for p in range(L):
            page = bt[2, p // 16]
            cb = oracle.chunk_bytes(d_h, lay["g"])
            kc, vc, km, vm = _unpack_chunk(paged[(page * h_kv + h) * cb:(page * h_kv + h + 1) * cb],
                                           d_h, lay["g"])
            c4, d4, m4, _ = oracle.int4_encode(W.bf16_bits_to_f32(k[h, p]), lay["g"])
            assert np.array_equal(kc[p % 16], c4) and np.array_equal(km[p % 16, :, 0], d4)
    # the other request slots' side blocks are untouched
    sb = oracle.side_block_bytes(d_h, S, R)
    assert np.all(side[: 2 * h_kv * sb] == CANARY)


def test_bad_arguments_set_status_and_write_nothing():
    lay, paged, side = _setup()
    h_kv, d_h = lay["h_kv"], lay["d_h"]
    bt = np.full((3, 4), -1, dtype=np.int32)
    bt[0] = [0, 99, -1, -1]
    k = np.zeros((4, h_kv, d_h), dtype=np.uint16)
    p0, s0 = paged.copy(), side.copy()
    st = oracle.quant_append(**lay, paged=paged, side=side, k_new=k, v_new=k,
                             tok_seq=np.array([5, 0, 0, 0]), tok_pos=np.array([0, 20, 40, 9]),
                             seq_lens=np.array([30, 0, 0], dtype=np.int32), block_table=bt)
    # seq 5 out of range; page 99 out of range; pos 40 beyond the length;
    # pos 9 on page-table entry 0 is valid and is written
    assert st == oracle.ST_BAD_SEQ | oracle.ST_BAD_PAGE | oracle.ST_BAD_POS
    cb = oracle.chunk_bytes(d_h, lay["g"])
    assert np.array_equal(paged[h_kv * cb:], p0[h_kv * cb:])
