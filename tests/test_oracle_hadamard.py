"""Pins for the oracle's Hadamard K-rotation (KV4-RL Sec. 3 eq. 3.4: a
normalized Hadamard H with H H^T = I leaves q.k unchanged when applied to both;
App. A.3 "Encoding and allocation": K and Q rotated after RoPE, V kept in its
own basis; App. D.4: K-only rotation retained).

Each check ties the oracle to something other than itself: scipy's Sylvester
construction, exact integer arithmetic, the fp32 error bound of the butterfly,
torch's bf16 rounding, and the orthogonality invariant.  A wrong sign or
partner index, a missing normalisation (the unnormalized transform is off by
sqrt(d)), rotating V, or skipping the rotation before one of the two encoders
fails at least one of them.
"""
import math

import numpy as np
import pytest
import scipy.linalg as sl
import torch

import oracle
from int8_kv_cache_kv4_gb300 import workloads as W

U32 = 2.0 ** -24          # unit roundoff of fp32
DIMS = [1, 2, 4, 8, 16, 32, 64, 128, 256]


def _bound(x, n):
    """Forward error bound of the fp32 butterfly plus the final scaling:
    log2(n) rounded additions on partial sums bounded by sum|x|, then one
    rounded multiply by a constant that is itself within U32 of 1/sqrt(n)."""
    s = np.abs(x.astype(np.float64)).sum(-1, keepdims=True)
    return (math.log2(n) + 3) * U32 * s / math.sqrt(n) * 1.01


@pytest.mark.parametrize("n", DIMS)
def test_unit_vectors_give_sylvester_rows(n):
    # H e_i is column i of the Sylvester matrix; every entry is +-fp32(1/sqrt n)
    c = np.float32(1.0 / math.sqrt(n))
    got = oracle.hadamard_f32(np.eye(n, dtype=np.float32))
    ref = (sl.hadamard(n).T * c).astype(np.float32)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("n", [8, 64, 128])
def test_integer_inputs_are_exact(n):
    # small integers: every butterfly sum is exact, so the result is the exact
    # integer product H x rounded once by the final scaling
    rng = np.random.default_rng(n)
    x = rng.integers(-300, 301, size=(20, n)).astype(np.float32)
    hx = x.astype(np.int64) @ sl.hadamard(n).T.astype(np.int64)
    ref = (hx.astype(np.float32) * np.float32(1.0 / math.sqrt(n))).astype(np.float32)
    assert np.array_equal(oracle.hadamard_f32(x), ref)


@pytest.mark.parametrize("n", [16, 64, 128, 256])
def test_matches_fp64_matrix_product_within_fp32_bound(n):
    rng = np.random.default_rng(100 + n)
    x = (rng.standard_normal((64, n)) * np.exp2(rng.integers(-8, 9, size=(64, 1)))).astype(np.float32)
    x[0, 5] = 300.0                       # an outlier channel
    ref = x.astype(np.float64) @ sl.hadamard(n).T / math.sqrt(n)
    err = np.abs(oracle.hadamard_f32(x).astype(np.float64) - ref)
    assert np.all(err <= _bound(x, n))


@pytest.mark.parametrize("n", [32, 128])
def test_involution_and_score_invariance(n):
    # H is symmetric and orthogonal: H(Hx) = x and (Hq).(Hk) = q.k (eq. 3.4)
    rng = np.random.default_rng(7 * n)
    q = rng.standard_normal((16, n)).astype(np.float32)
    k = rng.standard_normal((16, n)).astype(np.float32)
    hq, hk = oracle.hadamard_f32(q), oracle.hadamard_f32(k)
    back = oracle.hadamard_f32(hq)
    assert np.all(np.abs(back - q) <= 2 * _bound(q, n))
    dots = (q.astype(np.float64) * k).sum(-1)
    rdots = (hq.astype(np.float64) * hk).sum(-1)
    scale = np.linalg.norm(q, axis=-1) * np.linalg.norm(k, axis=-1)
    assert np.all(np.abs(rdots - dots) <= 8 * (math.log2(n) + 3) * U32 * scale)
    # the norm is kept too, so an unnormalized transform (off by sqrt n) fails
    np.testing.assert_allclose(np.linalg.norm(hk, axis=-1), np.linalg.norm(k, axis=-1),
                               rtol=1e-5)


def test_bf16_query_rotation_is_nearest_even_rounding():
    q = W.q_numpy(3, 4, 32, 128)
    got = oracle.hadamard_bf16(q)
    f = oracle.hadamard_f32(W.bf16_bits_to_f32(q))
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert got.dtype == np.uint16 and np.array_equal(got, ref)


# ------------------------------------------------- the rotation in the cache

def _seq(seed, h_kv, L, d_h):
    outl = W.outlier_channels(seed, h_kv, d_h)
    return W.kv_numpy_block(seed, 0, h_kv, L, d_h, outl)


@pytest.mark.parametrize("g", [32, 128])
def test_rotation_applies_to_k_before_both_encoders_and_never_to_v(g):
    h_kv, L, d_h, S, R = 2, 48, 128, 4, 12
    k, v = _seq(31, h_kv, L, d_h)
    kh0, vh0, st0 = oracle.dequant_seq(k, v, g=g, S=S, R=R)
    kh, vh, st = oracle.dequant_seq(k, v, g=g, S=S, R=R, rotate_k=True)
    assert st == 0 and st0 == 0
    assert np.array_equal(vh, vh0)                       # V stays in its basis
    # the stored K approximates the rotated source H k, not k itself
    hk = W.bf16_bits_to_f32(k).astype(np.float64) @ sl.hadamard(d_h).T / math.sqrt(d_h)
    for p in range(L):
        e = np.abs(kh[:, p] - hk[:, p])
        if p < S or p >= L - R:
            # INT8: half a step of max|Hk|/127, the fp16 scale rounded up
            tol = np.abs(hk[:, p]).max(-1, keepdims=True) / 127 * (0.5 + 2 ** -10) + 1e-6
        else:
            # INT4: half a step of the group range / 15 (plus fp16 metadata)
            grp = hk[:, p].reshape(h_kv, d_h // g, g)
            rng_ = (grp.max(-1) - grp.min(-1)) / 15 * (1 + 2 ** -9)
            tol = np.repeat(rng_ / 2 + np.abs(grp).max(-1) * 2 ** -10, g, axis=-1) + 1e-6
        assert np.all(e <= tol), p
        # and it is far from the unrotated source (the outlier is spread out)
        assert np.abs(kh[:, p] - W.bf16_bits_to_f32(k[:, p])).max() > 10 * tol.max()


def test_rotated_decode_approximates_unrotated_attention():
    # with q rotated by the same matrix, rotated-K attention approximates the
    # exact attention of the unrotated bf16 cache (eq. 3.4); attending with an
    # unrotated q does not
    h_q, h_kv, d_h, L = 8, 2, 128, 64
    k, v = _seq(41, h_kv, L, d_h)
    q = W.q_numpy(42, 1, h_q, d_h)[0]
    sc = 1 / math.sqrt(d_h)
    kf = W.bf16_bits_to_f32(k).astype(np.float64)
    vf = W.bf16_bits_to_f32(v).astype(np.float64)
    exact, exact_lse = oracle.attend(q, kf, vf, sc)
    qr = oracle.hadamard_bf16(q)
    # every position protected (INT8): close to the exact attention
    out, lse, st = oracle.decode_seq(qr, k, v, g=32, S=4, R=60, sm_scale=sc, rotate_k=True)
    assert st == 0
    np.testing.assert_allclose(out, exact, atol=0.05 * np.abs(exact).max(), rtol=0)
    np.testing.assert_allclose(lse, exact_lse, atol=0.05, rtol=0)
    bad, _, _ = oracle.decode_seq(q, k, v, g=32, S=4, R=60, sm_scale=sc, rotate_k=True)
    assert np.abs(bad - exact).max() > 10 * np.abs(out - exact).max()
    # mixed INT4/INT8 cache with outlier channels in K: the rotation spreads
    # them over the head, so the INT4 error shrinks (the reason for rotating)
    for g in (32, 128):
        rot, rlse, _ = oracle.decode_seq(qr, k, v, g=g, S=4, R=16, sm_scale=sc, rotate_k=True)
        plain, plse, _ = oracle.decode_seq(q, k, v, g=g, S=4, R=16, sm_scale=sc)
        assert np.abs(rot - exact).max() < 0.5 * np.abs(plain - exact).max()
        assert np.abs(rlse - exact_lse).max() < 0.5 * np.abs(plse - exact_lse).max()


def test_packed_append_with_rotation_matches_rotated_dequant():
    # the packed writer and the per-sequence reader agree on the rotation
    h_kv, d_h, g, S, R, L = 2, 128, 32, 4, 16, 40
    k, v = _seq(51, h_kv, L, d_h)
    out = {}
    for rot in (False, True):
        kh, vh, _ = oracle.dequant_seq(k, v, g=g, S=S, R=R, rotate_k=rot)
        out[rot] = kh
    assert not np.array_equal(out[False], out[True])
    # bytes: appending with rotation equals appending without it once K is
    # replaced by a vector whose fp32 rotation is exactly representable in
    # bf16: at d = 64, 1/sqrt(d) = 1/8, so two scaled unit vectors rotate to
    # (+-a +- b) / 8 exactly
    d_h = 64
    e = np.zeros((1, h_kv, d_h), dtype=np.float32)
    e[0, :, 3] = 2.0 ** 6
    e[0, 1, 10] = -2.0 ** 4
    he = oracle.hadamard_f32(e)
    ref = e[0].astype(np.float64) @ sl.hadamard(d_h).T / 8
    assert np.array_equal(he[0], ref) and np.array_equal(W.bf16_bits_to_f32(W.f32_to_bf16_bits(he)), he)
    vb = W.f32_to_bf16_bits(np.ones((1, h_kv, d_h), dtype=np.float32))
    res = []
    for kin, rot in ((W.f32_to_bf16_bits(e), True), (W.f32_to_bf16_bits(he), False)):
        paged = np.zeros(4 * h_kv * oracle.chunk_bytes(d_h, g), dtype=np.uint8)
        side = np.zeros(h_kv * oracle.side_block_bytes(d_h, S, R), dtype=np.uint8)
        st = oracle.quant_append(h_kv=h_kv, d_h=d_h, g=g, S=S, R=R, max_seqs=1, num_pages=4,
                                 max_pages_per_seq=4, paged=paged, side=side, k_new=kin,
                                 v_new=vb, tok_seq=np.zeros(1, np.int32),
                                 tok_pos=np.zeros(1, np.int32), seq_lens=np.ones(1, np.int32),
                                 block_table=np.arange(4, dtype=np.int32), rotate_k=rot)
        assert st == 0
        res.append((paged.copy(), side.copy()))
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])
