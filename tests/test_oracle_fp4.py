"""Pins for the oracle's FP4 probe formats (KV4-RL App. D.4, Fig. A4(c)):
E2M1 and E4M3 element rounding against brute force over every representable
value and against torch's float8_e4m3fn conversion; the MXFP4 shared scale
against its closed form; NVFP4's two-level scales against their defining
bounds; the storage cost the pages print (tests/golden/); the packed probe
cache parsed back; the K-only rotation; and the probe attention against exact
attention.  A wrong tie rule, a missing saturation, a block of the wrong size
or a global scale off by the E4M3 range fails at least one of them."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from int8_kv_cache_kv4_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _e2m1_from_bits(c):
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    v = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
    return -v if s else v


def _e4m3_from_bits(c):
    s, e, m = (c >> 7) & 1, (c >> 3) & 15, c & 7
    if e == 15 and m == 7:
        return math.nan
    v = m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return -v if s else v


def test_element_value_tables_from_bit_fields():
    for c in range(16):
        assert oracle.e2m1_value(c) == _e2m1_from_bits(c)
    for c in range(256):
        a, b = oracle.e4m3_value(c), _e4m3_from_bits(c)
        assert (math.isnan(a) and math.isnan(b)) or a == b, c
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e2m1_value(7) == 6.0


def _nearest_code(y, values, codes):
    """Brute force: the code of the value nearest |y|, ties to the even code."""
    d = np.abs(values - abs(y))
    best = np.flatnonzero(d == d.min())
    if len(best) > 1:
        best = [b for b in best if codes[b] % 2 == 0]
    return codes[best[0]]


def test_e2m1_rounding_brute_force_with_midpoints():
    vals = np.array([_e2m1_from_bits(c) for c in range(8)])
    mids = (vals[1:] + vals[:-1]) / 2
    rng = np.random.default_rng(1)
    ys = np.concatenate([vals, mids, np.nextafter(mids, 0), np.nextafter(mids, 10),
                         rng.uniform(0, 6, 2000), [5.999, 6.0, 6.5, 100.0, 1e30]]).astype(np.float32)
    ys = np.concatenate([ys, -ys])
    got = oracle.e2m1_round(ys)
    for y, c in zip(ys, got):
        want = 7 if abs(y) >= 6 else _nearest_code(float(y), vals, np.arange(8))
        assert (c & 7) == want and (c >> 3) == (1 if np.signbit(y) else 0), (y, c)


def test_e4m3_rounding_brute_force_and_torch():
    vals = np.array([_e4m3_from_bits(c) for c in range(0x7F)])
    mids = (vals[1:] + vals[:-1]) / 2
    rng = np.random.default_rng(2)
    ts = np.concatenate([vals, mids, np.exp2(rng.uniform(-12, 9, 3000)),
                         [447.9, 448.0, 460.0, 500.0, 1e6]]).astype(np.float32)
    got = oracle.e4m3_round(ts)
    for t, c in zip(ts, got):
        want = 0x7E if t >= 448 else _nearest_code(float(t), vals, np.arange(0x7F))
        assert c == want, (t, c, want)
    # torch's float8_e4m3fn rounds to nearest even (it saturates only below 464)
    inr = ts[ts < 464]
    ref = torch.from_numpy(inr).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_round(inr), ref)


def test_mxfp4_scale_closed_form_and_error():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((200, 128)) * np.exp2(rng.integers(-20, 20, (200, 1)))).astype(np.float32)
    x[0, :32] = 0.0                                       # an all-zero block
    codes, bs, g, st = oracle.fp4_encode(x, oracle.MXFP4)
    assert st == 0 and bs.shape == (200, 4) and np.all(g == 0)
    amax = np.abs(x.reshape(200, 4, 32)).max(-1)
    _, e2 = np.frexp(amax)
    E = np.where(amax > 0, e2 - 1 - 2, -127)
    assert np.array_equal(bs.astype(int) - 127, E)
    X = np.exp2(E.astype(np.float64))
    r = amax / X
    assert np.all((r[amax > 0] >= 4) & (r[amax > 0] < 8))
    y = oracle.fp4_decode(codes, bs, g, oracle.MXFP4).reshape(200, 4, 32).astype(np.float64)
    xs = x.reshape(200, 4, 32).astype(np.float64)
    # half an E2M1 step (1 above 4, i.e. 2 X / 2), or the clip at 6 X
    bound = np.maximum(X[..., None], np.abs(xs) - 6 * X[..., None])
    assert np.all(np.abs(y - xs) <= bound + 1e-30)
    assert np.all(y[0, 0] == 0)


def test_nvfp4_two_level_scales():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((300, 128)) * np.exp2(rng.integers(-12, 12, (300, 1)))).astype(np.float32)
    x[:, 5] *= 30                                         # an outlier channel
    codes, bs, g, st = oracle.fp4_encode(x, oracle.NVFP4)
    assert st == 0 and bs.shape == (300, 8)
    amax = np.abs(x).max(-1)
    assert np.array_equal(g, (amax / np.float32(2688)).astype(np.float32))
    # the block holding the vector's maximum gets E4M3's largest scale, 448
    top = np.abs(x).reshape(300, 8, 16).max(-1).argmax(-1)
    assert np.all(bs[np.arange(300), top] == 0x7E)
    # reconstruction: within half an E2M1 step of x / e_b, times e_b, or the clip
    eb = np.array([[oracle.e4m3_value(c) for c in row] for row in bs], dtype=np.float32) * g[:, None]
    eb = np.repeat(eb.astype(np.float64), 16, axis=1)
    y = oracle.fp4_decode(codes, bs, g, oracle.NVFP4).astype(np.float64)
    a = np.abs(x.astype(np.float64)) / eb
    half = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0)) * eb
    bound = np.maximum(half, np.abs(x) - 6 * eb) * (1 + 1e-6)
    assert np.all(np.abs(y - x) <= bound)


def test_exactly_representable_vectors_round_trip():
    # MXFP4: E2M1 values times one power of two per block reconstruct exactly
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 16, (10, 64))
    codes[:, ::32] = 7                                    # each block reaches 6 X
    vals = np.array([_e2m1_from_bits(int(c)) for c in codes.ravel()]).reshape(10, 64)
    x = (vals * np.repeat(np.exp2(rng.integers(-8, 8, (10, 2))), 32, axis=1)).astype(np.float32)
    c, bs, g, _ = oracle.fp4_encode(x, oracle.MXFP4)
    assert np.array_equal(oracle.fp4_decode(c, bs, g, oracle.MXFP4), x)


def test_storage_bits_per_element_golden():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "fp4_bits_per_element.txt"))
            if l.strip() and not l.startswith("#")]
    x = np.random.default_rng(6).standard_normal((1, 128)).astype(np.float32)
    for name, bits_s, gbits_s in rows:
        fmt = {"nvfp4": oracle.NVFP4, "mxfp4": oracle.MXFP4}[name]
        codes, bs, g, _ = oracle.fp4_encode(x, fmt)
        assert codes.max() < 16                          # 4-bit codes
        gbits = 32 / 128 if fmt == oracle.NVFP4 else 0.0  # one fp32 per vector
        bits = 4 + bs.shape[-1] * 8 / 128 + gbits
        assert bits == pytest.approx(float(bits_s)) and gbits == pytest.approx(float(gbits_s))


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP4])
def test_packed_probe_cache_parses_back(fmt):
    h_kv, d_h, P = 2, 128, 3
    outl = W.outlier_channels(7, h_kv, d_h)
    k, v = W.kv_numpy_block(7, 0, h_kv, 20, d_h, outl)
    rb = oracle.fp4_row_bytes(d_h)
    cache = np.full(P * h_kv * 2 * 16 * rb, 0xA5, dtype=np.uint8)
    bt = np.array([[2, 0]], dtype=np.int32)
    pos = np.array([0, 5, 17], dtype=np.int32)
    st = oracle.fp4_append(h_kv=h_kv, d_h=d_h, fmt=fmt, rotate_k=True, max_seqs=1, num_pages=P,
                           max_pages_per_seq=2, cache=cache,
                           k_new=np.ascontiguousarray(k[:, pos].transpose(1, 0, 2)),
                           v_new=np.ascontiguousarray(v[:, pos].transpose(1, 0, 2)),
                           tok_seq=np.zeros(3, np.int32), tok_pos=pos,
                           seq_lens=np.array([20], np.int32), block_table=bt)
    assert st == 0
    rows = cache.reshape(P, h_kv, 2, 16, rb)
    nb = d_h // 16 if fmt == oracle.NVFP4 else d_h // 32
    touched = np.zeros((P, 16), bool)
    for i, p in enumerate(pos):
        page, slot = bt[0, p // 16], p % 16
        touched[page, slot] = True
        for h in range(h_kv):
            for kv, src in ((0, k), (1, v)):
                x = W.bf16_bits_to_f32(src[h, p])
                if kv == 0:
                    x = oracle.hadamard_f32(x)                # K only, before encoding
                codes, bs, g, _ = oracle.fp4_encode(x, fmt)
                row = rows[page, h, kv, slot]
                assert np.array_equal(row[: d_h // 2] & 15, codes[0::2])
                assert np.array_equal(row[: d_h // 2] >> 4, codes[1::2])
                assert np.array_equal(row[d_h // 2: d_h // 2 + nb], bs)
                if fmt == oracle.NVFP4:
                    assert row[d_h // 2 + 12: d_h // 2 + 16].view(np.float32)[0] == g
                else:
                    assert np.all(row[d_h // 2 + nb:] == 0xA5)
    assert np.all(rows.transpose(0, 3, 1, 2, 4)[~touched] == 0xA5)   # no other slot written


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP4])
def test_probe_attention_near_exact_and_rotation_is_k_only(fmt):
    h_q, h_kv, d_h, L = 8, 2, 128, 48
    outl = W.outlier_channels(8, h_kv, d_h)
    k, v = W.kv_numpy_block(8, 0, h_kv, L, d_h, outl)
    q = W.q_numpy(9, 1, h_q, d_h)[0]
    sc = 1 / math.sqrt(d_h)
    exact, else_ = oracle.attend(q, W.bf16_bits_to_f32(k).astype(np.float64),
                                 W.bf16_bits_to_f32(v).astype(np.float64), sc)
    out, lse, st = oracle.fp4_decode_seq(q, k, v, fmt=fmt, sm_scale=sc)
    assert st == 0
    assert np.abs(out - exact).max() < 0.4 * np.abs(exact).max()
    kh0, vh0, _ = oracle.fp4_dequant_seq(k, v, fmt=fmt)
    kh1, vh1, _ = oracle.fp4_dequant_seq(k, v, fmt=fmt, rotate_k=True)
    assert np.array_equal(vh0, vh1) and not np.array_equal(kh0, kh1)
    # the operands are bf16 values
    assert np.array_equal(W.bf16_bits_to_f32(W.f32_to_bf16_bits(kh1.astype(np.float32))), kh1)
    # with the rotated query, rotated-K attention is the same quantity
    outr, _, _ = oracle.fp4_decode_seq(oracle.hadamard_bf16(q), k, v, fmt=fmt, sm_scale=sc,
                                       rotate_k=True)
    assert np.abs(outr - exact).max() < 0.4 * np.abs(exact).max()
