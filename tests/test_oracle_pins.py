"""Pins for the CPU oracle: each check ties an oracle function to something
other than itself -- a library routine, exact rational arithmetic, a closed
form, an invariant the paper states, brute force, or a number the paper
prints (tests/golden/).  A plausible mistake in the oracle (a wrong rounding
direction, a dropped offset, a swapped nibble, an off-by-one in the protected
window, a wrong merge weight) fails at least one of these.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from int8_kv_cache_kv4_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

ALL_F16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _finite_f16_table():
    with np.errstate(invalid="ignore"):
        v = ALL_F16.view(np.float16).astype(np.float64)
    ok = np.isfinite(v)
    bits = ALL_F16[ok]
    vals = v[ok]
    order = np.argsort(vals, kind="stable")
    vals, bits = vals[order], bits[order]
    # collapse -0/+0 to one entry with +0 bits
    keep = np.ones(len(vals), dtype=bool)
    keep[1:] = vals[1:] != vals[:-1]
    return vals[keep], bits[keep]


F16_VALS, F16_BITS = _finite_f16_table()


def _rand_f32(n, seed):
    rng = np.random.default_rng(seed)
    mag = np.exp2(rng.uniform(-28, 17, size=n))
    x = (mag * rng.choice([-1.0, 1.0], size=n)).astype(np.float32)
    return x


# ----------------------------------------------------------- fp16 rounding

def test_f16_to_f32_matches_numpy_all_patterns():
    got = oracle.f16_to_f32(ALL_F16)
    ref = ALL_F16.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f32_to_f16_nearest_even_matches_numpy():
    x = np.concatenate([_rand_f32(200000, 1),
                        # exact ties between adjacent fp16 values
                        ((F16_VALS[1:-1] + F16_VALS[2:]) / 2).astype(np.float32),
                        np.array([65504, 65519.99, 65520, 1e6, -65520, 2**-25, 2**-26, 3 * 2**-26,
                                  0.0, -0.0], dtype=np.float32)])
    got = oracle.f32_to_f16(x, oracle.RNE)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("mode", [oracle.DOWN, oracle.UP])
def test_f32_to_f16_directed_is_bracketing_neighbour(mode):
    x = _rand_f32(100000, 2)
    x = x[np.abs(x) <= 65504]
    got = oracle.f32_to_f16(x, mode).view(np.float16).astype(np.float64)
    xd = x.astype(np.float64)
    if mode == oracle.DOWN:
        idx = np.searchsorted(F16_VALS, xd, side="right") - 1
        ref = F16_VALS[idx]
    else:
        idx = np.searchsorted(F16_VALS, xd, side="left")
        ref = F16_VALS[idx]
    assert np.array_equal(got, ref)


def test_f32_to_f16_directed_overflow():
    x = np.array([70000.0, -70000.0], dtype=np.float32)
    up = oracle.f32_to_f16(x, oracle.UP).view(np.float16).astype(np.float64)
    dn = oracle.f32_to_f16(x, oracle.DOWN).view(np.float16).astype(np.float64)
    assert up[0] == np.inf and up[1] == -65504.0
    assert dn[0] == 65504.0 and dn[1] == -np.inf


# ------------------------------------------------- directed fp32 operations

def _smallest_f32_ge(q: Fraction) -> np.float32:
    f = np.float32(float(q))  # nearest double -> nearest float, then fix up
    while Fraction(float(f)) < q:
        f = np.nextafter(f, np.float32(np.inf))
    while Fraction(float(np.nextafter(f, np.float32(-np.inf)))) >= q:
        f = np.nextafter(f, np.float32(-np.inf))
    return f


def test_directed_sub_div_against_exact_rationals():
    rng = np.random.default_rng(3)
    a = rng.standard_normal(3000).astype(np.float32) * np.float32(7)
    b = rng.standard_normal(3000).astype(np.float32)
    b[np.abs(b) < 1e-3] = np.float32(0.5)
    su = oracle.sub_dir(a, b, oracle.UP)
    du = oracle.div_dir(a, b, oracle.UP)
    for i in range(0, 3000, 7):
        assert su[i] == _smallest_f32_ge(Fraction(float(a[i])) - Fraction(float(b[i])))
        assert du[i] == _smallest_f32_ge(Fraction(float(a[i])) / Fraction(float(b[i])))
    # round-to-nearest matches numpy's IEEE float32 arithmetic
    assert np.array_equal(oracle.sub_dir(a, b, oracle.RNE), (a - b).astype(np.float32))
    assert np.array_equal(oracle.div_dir(a, b, oracle.RNE), (a / b).astype(np.float32))


# ---------------------------------------------------------------- INT4 encode

def _groups(seed, n, g):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, g)).astype(np.float32)
    x[: n // 4] *= 8.0                                     # outlier-scale groups
    x[n // 4: n // 2] *= np.float32(1e-3)                  # tiny values
    x[n // 2: n // 2 + 8] = np.float32(0.3)                # constant groups
    x[n // 2 + 8: n // 2 + 16, 3] *= 300.0                 # one huge element
    return W.bf16_bits_to_f32(W.f32_to_bf16_bits(x))       # bf16 inputs


@pytest.mark.parametrize("g", [8, 32, 64, 128])
def test_int4_error_bound_and_metadata_bracket(g):
    x = _groups(4, 2000, g)
    codes, d16, m16, st = oracle.int4_encode(x, g)
    assert st == 0
    assert codes.max() <= 15
    D = d16.view(np.float16).astype(np.float64)[:, 0]
    M = m16.view(np.float16).astype(np.float64)[:, 0]
    xd = x.astype(np.float64)
    mn, mx = xd.min(1), xd.max(1)
    # m is the fp16 value rounded down from the group minimum (tight)
    assert np.all(M <= mn)
    nxt = np.nextafter(m16.view(np.float16)[:, 0], np.float16(np.inf)).astype(np.float64)
    assert np.all(nxt > mn)
    # the lattice covers the group: m + 15*Delta >= max, so no code clamps
    assert np.all(M + 15 * D >= mx)
    # reconstruction error <= Delta/2 (plus fp32 quotient rounding)
    rec = D[:, None] * codes + M[:, None]
    err = np.abs(xd - rec)
    assert np.all(err <= D[:, None] * (0.5 + 2 ** -20) + 1e-30)
    # codes are monotone in x within a group
    for r in range(0, 2000, 13):
        o = np.argsort(xd[r], kind="stable")
        assert np.all(np.diff(codes[r][o].astype(int)) >= 0)


def test_int4_closed_form_lattice():
    # x = m + k*Delta with m, Delta exact in fp16 and x exact in bf16
    m, D = -1.0, 0.125
    k = np.array([0, 15, 3, 7, 8, 1, 14, 2, 9, 11, 5, 4, 6, 10, 12, 13], dtype=np.int64)
    x = (m + D * k).astype(np.float32)[None, :]
    codes, d16, m16, st = oracle.int4_encode(x, 16)
    assert st == 0
    assert np.array_equal(codes[0], k.astype(np.uint8))
    assert float(d16.view(np.float16)[0, 0]) == D and float(m16.view(np.float16)[0, 0]) == m


def test_int4_min_to_zero_and_max_to_top_for_bf16_inputs():
    x = _groups(5, 500, 32)[: 250]   # outlier and unit-scale groups: fp16-exact minimum
    codes, d16, m16, _ = oracle.int4_encode(x, 32)
    amin = np.argmin(x, axis=1)
    amax = np.argmax(x, axis=1)
    r = np.arange(len(x))
    assert np.all(codes[r, amin] == 0)
    assert np.all(codes[r, amax] >= 14)


def test_int4_constant_group_and_nonfinite():
    # constant group of an fp16-exact value: Delta = 0, codes 0, m = value
    x = np.full((1, 32), 0.375, dtype=np.float32)
    codes, d16, m16, st = oracle.int4_encode(x, 32)
    assert st == 0 and d16[0, 0] == 0 and np.all(codes == 0)
    assert float(m16.view(np.float16)[0, 0]) == 0.375
    # constant group of a value between fp16 neighbours: one shared code
    x = np.full((1, 32), 0.3, dtype=np.float32)
    codes, d16, m16, st = oracle.int4_encode(x, 32)
    assert st == 0 and len(set(codes[0].tolist())) == 1
    x = np.zeros((2, 32), dtype=np.float32)
    x[1, 5] = np.inf
    codes, d16, m16, st = oracle.int4_encode(x, 32)
    assert st == oracle.ST_NONFINITE
    assert np.all(codes[1] == 0) and d16[1, 0] == 0 and m16[1, 0] == 0
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0] = -1e5            # below the fp16 range: offset overflows
    _, _, _, st = oracle.int4_encode(x, 32)
    assert st == oracle.ST_NONFINITE


def test_storage_bits_per_element_golden():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "storage_bits_per_element.txt"))
            if l.strip() and not l.startswith("#")]
    for g_s, bits_s in rows:
        g = int(g_s)
        d_h = 128
        # one K (or V) chunk half: 16 slots of codes plus metadata
        per_side_bytes = oracle.chunk_bytes(d_h, g) / 2
        bits = per_side_bytes * 8 / (16 * d_h)
        assert bits == pytest.approx(float(bits_s), abs=1e-12)


def test_bf16_kv_bytes_per_token_golden():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "kv_bytes_per_token.txt"))
            if l.strip() and not l.startswith("#")]
    for name, layers, heads, d_h, nbytes in rows:
        assert 2 * int(layers) * int(heads) * int(d_h) * 2 == int(nbytes), name


# ---------------------------------------------------------------- INT8 encode

def test_int8_invariants():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3000, 128)).astype(np.float32)
    x[:500] *= 8
    x[500:600] *= 1e-4
    codes, s16, st = oracle.int8_encode(x)
    assert st == 0
    s = s16.view(np.float16).astype(np.float64)
    a = np.abs(x.astype(np.float64)).max(1)
    assert np.all(s >= a / 127)           # scale rounded up: no clamping
    assert np.all(np.abs(codes.astype(int)) <= 127)
    err = np.abs(x - s[:, None] * codes)
    assert np.all(err <= s[:, None] * (0.5 + 2 ** -20))
    c2, s2, _ = oracle.int8_encode(-x)
    assert np.array_equal(s2, s16) and np.array_equal(c2.astype(int), -codes.astype(int))


def test_int8_closed_form():
    x = np.zeros((2, 128), dtype=np.float32)
    x[0, 7] = 127 * 2 ** -5
    x[0, 9] = -63 * 2 ** -5
    codes, s16, st = oracle.int8_encode(x)
    assert float(s16.view(np.float16)[0]) == 2 ** -5
    assert codes[0, 7] == 127 and codes[0, 9] == -63 and np.count_nonzero(codes[0]) == 2
    assert s16[1] == 0 and np.all(codes[1] == 0)


# ----------------------------------------------------------- protection rule

def test_protected_set_worked_example():
    # L = 20, first s = 3 and most recent w = 5 positions (KV4-RL Sec. 5.2)
    got = [p for p in range(20) if oracle.is_protected(p, 20, 3, 5)]
    assert got == [0, 1, 2, 15, 16, 17, 18, 19]
    # overlap when L <= S + R: everything protected, at most S + R positions
    assert all(oracle.is_protected(p, 7, 3, 5) for p in range(7))
    for L in range(0, 40):
        n = sum(oracle.is_protected(p, L, 4, 6) for p in range(L))
        assert n == min(L, 10)
    # ring slots of the recent window are distinct
    L, S, R = 100, 4, 16
    slots = {oracle.side_slot(p, S, R) for p in range(L) if oracle.is_protected(p, L, S, R)}
    assert len(slots) == S + R and slots == set(range(S + R))


# ------------------------------------------------------------------ attention

def _seq(seed, h_kv, L, d_h):
    outl = W.outlier_channels(seed, h_kv, d_h)
    return W.kv_numpy_block(seed, 0, h_kv, L, d_h, outl)


def _textbook(q, kh, vh, sm_scale):
    """numpy softmax(q K^T * scale) V for each query head."""
    qf = W.bf16_bits_to_f32(q).astype(np.float64)
    h_q = qf.shape[0]
    h_kv = kh.shape[0]
    G = h_q // h_kv
    out = np.empty((h_q, kh.shape[2]))
    lse = np.empty(h_q)
    for j in range(h_q):
        s = kh[j // G] @ qf[j] * sm_scale
        m = s.max()
        w = np.exp(s - m)
        out[j] = (w / w.sum()) @ vh[j // G]
        lse[j] = m + np.log(w.sum())
    return out, lse


@pytest.mark.parametrize("L", [1, 2, 5, 8])
@pytest.mark.parametrize("S,R", [(0, 0), (1, 2), (4, 64)])
def test_attention_brute_force_small(L, S, R):
    h_q, h_kv, d_h = 8, 2, 64
    k, v = _seq(7 + L, h_kv, L, d_h)
    q = W.q_numpy(8, 1, h_q, d_h)[0]
    sc = 1 / math.sqrt(d_h)
    out, lse, st = oracle.decode_seq(q, k, v, g=32, S=S, R=R, sm_scale=sc)
    kh, vh, _ = oracle.dequant_seq(k, v, g=32, S=S, R=R)
    ref, rlse = _textbook(q, kh, vh, sc)
    assert st == 0
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rlse, rtol=0, atol=1e-12)


def test_dequant_regions_against_encoders():
    # protected positions decode the INT8 entry of the source vector,
    # the others the INT4 entry (Sec. 5.3: disjoint regions)
    h_kv, L, d_h, S, R = 2, 40, 64, 3, 5
    k, v = _seq(9, h_kv, L, d_h)
    kh, vh, _ = oracle.dequant_seq(k, v, g=16, S=S, R=R)
    x = W.bf16_bits_to_f32(k)
    c8, s8, _ = oracle.int8_encode(x)
    c4, d4, m4, _ = oracle.int4_encode(x, 16)
    for h in range(h_kv):
        for p in range(L):
            if p < S or p >= L - R:
                ref = s8[h, p].view(np.float16).astype(np.float64) * c8[h, p]
            else:
                ref = (np.repeat(d4[h, p].view(np.float16).astype(np.float64), 16) * c4[h, p]
                       + np.repeat(m4[h, p].view(np.float16).astype(np.float64), 16))
            assert np.array_equal(kh[h, p], ref), (h, p)


def test_all_int8_when_protection_covers_sequence():
    # S + R >= L reduces to plain INT8 attention
    h_q, h_kv, d_h, L = 8, 2, 128, 30
    k, v = _seq(10, h_kv, L, d_h)
    q = W.q_numpy(11, 1, h_q, d_h)[0]
    sc = 1 / math.sqrt(d_h)
    out, lse, _ = oracle.decode_seq(q, k, v, g=32, S=4, R=26, sm_scale=sc)
    ck, sk, _ = oracle.int8_encode(W.bf16_bits_to_f32(k))
    cv, sv, _ = oracle.int8_encode(W.bf16_bits_to_f32(v))
    kh = sk.view(np.float16).astype(np.float64)[..., None] * ck
    vh = sv.view(np.float16).astype(np.float64)[..., None] * cv
    ref, rlse = _textbook(q, kh, vh, sc)
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=0)
    # and S = R = 0 is plain INT4 attention
    out4, _, _ = oracle.decode_seq(q, k, v, g=32, S=0, R=0, sm_scale=sc)
    c4, d4, m4, _ = oracle.int4_encode(W.bf16_bits_to_f32(k), 32)
    e4, f4, n4, _ = oracle.int4_encode(W.bf16_bits_to_f32(v), 32)
    up = lambda a: np.repeat(a.view(np.float16).astype(np.float64), 32, axis=-1)
    ref4, _ = _textbook(q, up(d4) * c4 + up(m4), up(f4) * e4 + up(n4), sc)
    np.testing.assert_allclose(out4, ref4, atol=1e-12, rtol=0)


def test_uniform_value_cache_gives_exact_value():
    h_q, h_kv, d_h, L = 8, 2, 128, 50
    k, _ = _seq(12, h_kv, L, d_h)
    val = np.float32(127 * 2 ** -7)     # exact in bf16, fp16, and as 127 * 2^-7
    v = W.f32_to_bf16_bits(np.full((h_kv, L, d_h), val, dtype=np.float32))
    q = W.q_numpy(13, 1, h_q, d_h)[0]
    out, _, _ = oracle.decode_seq(q, k, v, g=32, S=4, R=8, sm_scale=0.3)
    np.testing.assert_allclose(out, float(val), rtol=0, atol=1e-14)


def test_single_position_and_zero_query():
    h_q, h_kv, d_h = 8, 2, 64
    k, v = _seq(14, h_kv, 1, d_h)
    q = W.q_numpy(15, 1, h_q, d_h)[0]
    out, lse, _ = oracle.decode_seq(q, k, v, g=32, S=0, R=0, sm_scale=0.1)
    _, vh, _ = oracle.dequant_seq(k, v, g=32, S=0, R=0)
    for j in range(h_q):
        np.testing.assert_array_equal(out[j], vh[j // 4, 0])
    # q = 0: uniform weights, output is the mean of the dequantized values
    k, v = _seq(16, h_kv, 33, d_h)
    q0 = np.zeros((h_q, d_h), dtype=np.uint16)
    out, lse, _ = oracle.decode_seq(q0, k, v, g=32, S=2, R=5, sm_scale=0.1)
    _, vh, _ = oracle.dequant_seq(k, v, g=32, S=2, R=5)
    for j in range(h_q):
        np.testing.assert_allclose(out[j], vh[j // 4].mean(0), atol=1e-13, rtol=0)
        assert lse[j] == pytest.approx(math.log(33), abs=1e-13)


def test_gqa_group_one_is_mha():
    h, d_h, L = 4, 64, 12
    k, v = _seq(17, h, L, d_h)
    q = W.q_numpy(18, 1, h, d_h)[0]
    out, lse, _ = oracle.decode_seq(q, k, v, g=32, S=1, R=3, sm_scale=0.125)
    for j in range(h):
        o1, l1, _ = oracle.decode_seq(q[j:j + 1], k[j:j + 1], v[j:j + 1], g=32, S=1, R=3,
                                      sm_scale=0.125)
        np.testing.assert_array_equal(out[j], o1[0])
        assert lse[j] == l1[0]


# --------------------------------------------------------------------- merge

def test_merge_two_regions_closed_form():
    # z4 = log 3, z8 = log 1 -> weights 3/4 and 1/4 (App. A.3 eq. A1)
    o4 = np.array([1.0, 2.0, -4.0])
    o8 = np.array([5.0, -2.0, 0.0])
    out, z = oracle.combine(np.stack([o4, o8]), np.array([math.log(3.0), 0.0]))
    np.testing.assert_allclose(out, 0.75 * o4 + 0.25 * o8, atol=1e-15)
    assert z == pytest.approx(math.log(4.0), abs=1e-15)
    # an empty region has weight zero
    out, z = oracle.combine(np.stack([o4, o8 * np.nan]), np.array([0.3, -np.inf]))
    np.testing.assert_allclose(out, o4, atol=1e-15)
    assert z == pytest.approx(0.3)
    out, z = oracle.combine(np.zeros((3, 4)), np.full(3, -np.inf))
    assert z == -np.inf and np.all(out == 0)


def test_merge_partition_invariance():
    h_q, h_kv, d_h, L = 8, 2, 64, 45
    k, v = _seq(19, h_kv, L, d_h)
    q = W.q_numpy(20, 1, h_q, d_h)[0]
    kh, vh, _ = oracle.dequant_seq(k, v, g=32, S=3, R=7)
    full, flse = oracle.attend(q, kh, vh, 0.125)
    rng = np.random.default_rng(21)
    for trial in range(5):
        cuts = sorted(set([0, L] + rng.integers(0, L, size=4).tolist()))
        cuts.insert(1, 0)  # an empty part
        parts_o, parts_z = [], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            o, z = oracle.attend(q, kh[:, a:b], vh[:, a:b], 0.125)
            parts_o.append(o)
            parts_z.append(z)
        parts_o = np.stack(parts_o)
        parts_z = np.stack(parts_z)
        for j in range(h_q):
            o, z = oracle.combine(parts_o[:, j], parts_z[:, j])
            np.testing.assert_allclose(o, full[j], atol=1e-12, rtol=0)
            assert z == pytest.approx(flse[j], abs=1e-12)
