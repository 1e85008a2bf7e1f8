"""The KV-concentration driver's schedules (host logic, no GPU): their step
averages converge to the oracle's closed forms (KV4-RL Prop. 4.1; App. C
eqs. A4-A8), and every response occupies its slot exactly as the pages
describe (contexts P .. P+L-1, refills before the next step, waves that end
with their longest response)."""
import numpy as np
import pytest

from oracle import concentration as C
from int8_kv_cache_kv4_gb300 import rollout as R
from int8_kv_cache_kv4_gb300 import workloads as W

SUP = np.array([1, 2, 3, 5, 13])
PMF = np.array([0.3, 0.25, 0.2, 0.15, 0.1])


def test_refill_averages_match_closed_forms():
    B, P = 8, 6
    s = R.refill_schedule(B, P, SUP, PMF, 40000, np.random.default_rng(1))
    a = s.averages()
    assert a["active"] == B
    assert a["volume_tokens"] == pytest.approx(C.refill_volume(P, SUP, PMF, B), rel=0.02)
    assert a["mean_context"] == pytest.approx(C.refill_mean_context(P, SUP, PMF), rel=0.02)
    assert a["decode_tokens"] == pytest.approx(a["volume_tokens"] + B)   # + the new token


def test_wave_averages_match_closed_forms():
    B, P = 8, 6
    s = R.wave_schedule(B, P, SUP, PMF, 5000, np.random.default_rng(2))
    a = s.averages()
    assert a["volume_tokens"] == pytest.approx(C.wave_volume(P, SUP, PMF, B), rel=0.02)
    assert a["active"] == pytest.approx(C.wave_occupancy(SUP, PMF, B), rel=0.02)
    assert a["mean_context"] == pytest.approx(C.wave_mean_context(P, SUP, PMF, B), rel=0.02)


def test_measured_concentration_ratio():
    B, P = 16, 3
    sup, pmf = W.lognormal_length_pmf(40, 0.8, 4, 300)
    r = R.refill_schedule(B, P, sup, pmf, 60000, np.random.default_rng(3))
    w = R.wave_schedule(B, P, sup, pmf, 600, np.random.default_rng(4))
    ratio = r.averages()["volume_tokens"] / w.averages()["volume_tokens"]
    assert ratio == pytest.approx(C.concentration(sup, pmf, B), rel=0.04)
    assert ratio > 1.5


def test_refill_slots_follow_their_responses():
    B, P = 5, 4
    s = R.refill_schedule(B, P, SUP, PMF, 300, np.random.default_rng(5), stationary=False)
    assert s.lens.min() >= P + 1
    for b in range(B):
        L, rid = s.lens[:, b], s.resp[:, b]
        starts = [0] + [t for t in range(1, s.steps) if rid[t] != rid[t - 1]]
        for t0, t1 in zip(starts, starts[1:] + [s.steps]):
            assert np.array_equal(L[t0:t1], P + 1 + np.arange(t1 - t0))   # contexts P, P+1, ...
            assert len(np.unique(rid[t0:t1])) == 1
            if t1 < s.steps:                                              # a complete response
                assert t1 - t0 in SUP
                pre = s.prefill[t1]
                assert [b, rid[t1], P] in pre.tolist()                    # refilled before step t1
    # non-stationary start: every slot starts a response at step 0 with its prompt
    assert sorted(s.prefill[0][:, 0].tolist()) == list(range(B))


def test_stationary_start_prefills_prompt_and_earlier_tokens():
    B, P = 200, 7
    s = R.refill_schedule(B, P, SUP, PMF, 1, np.random.default_rng(6))
    pre = s.prefill[0]
    assert np.array_equal(pre[:, 0], np.arange(B))
    assert np.array_equal(pre[:, 2] + 1, s.lens[0])           # P + age written, then the new token
    # ages are spread over 0..L*-1 of length-biased lengths: mean age = E[L(L-1)] / (2 E[L])
    big = R.refill_schedule(20000, 0, SUP, PMF, 1, np.random.default_rng(7))
    mu, m2 = C.moments(SUP, PMF)
    assert (big.lens[0] - 1).mean() == pytest.approx(m2 / (2 * mu), rel=0.05)


def test_waves_end_with_their_longest_response():
    B, P = 6, 2
    s = R.wave_schedule(B, P, SUP, PMF, 30, np.random.default_rng(8))
    starts = [t for t in range(s.steps) if len(s.prefill[t])]
    assert len(starts) == 30 and starts[0] == 0
    for t0, t1 in zip(starts, starts[1:] + [s.steps]):
        blk = s.lens[t0:t1]
        assert (blk[-1] > 0).any()                 # the longest response runs to the end
        for b in range(B):
            n = int((blk[:, b] > 0).sum())
            assert np.array_equal(blk[:n, b], P + 1 + np.arange(n)) and np.all(blk[n:, b] == 0)


def test_decode_bytes_counts_regions():
    # one slot of 200 positions with S + R = 132: 132 INT8 + 68 INT4 token-heads
    b = R.decode_bytes(np.array([[200, 0]]), h_q=32, h_kv=8, d_h=128, group=32, sink=4, recent=128)
    assert b[0] == 8 * (132 * 260 + 68 * 160) + 13 * 4 + 32 * 128 * 4


@pytest.mark.parametrize("kind", ["refill", "waves"])
def test_chunk_plan_addresses_stay_inside_its_buffers(kind):
    # what drive() hands the C ABI per step: every (first row, count) and array
    # offset lies inside the chunk's buffers and holds the step's tokens
    B, P = 6, 9
    rng = np.random.default_rng(9)
    s = (R.refill_schedule(B, P, SUP, PMF, 40, rng) if kind == "refill"
         else R.wave_schedule(B, P, SUP, PMF, 4, rng))
    for c0 in range(0, s.steps, 7):
        c1 = min(s.steps, c0 + 7)
        rows, ints, plan = R._plan_chunk(s, c0, c1)
        assert len(plan) == c1 - c0
        for i, ent in enumerate(plan):
            t = c0 + i
            (r0, n_pre), (r1, n_tok), off = ent["pre"], ent["tok"], ent["off"]
            assert 0 <= r0 and r0 + n_pre == r1 and r1 + n_tok <= len(rows)
            sizes = [n_pre, n_pre, B, n_tok, n_tok, B]
            for k in range(6):
                assert 0 <= off[k] and off[k] + sizes[k] <= len(ints)
            pseq, ppos = ints[off[0]:off[0] + n_pre], ints[off[1]:off[1] + n_pre]
            plens = ints[off[2]:off[2] + B]
            tseq, tpos = ints[off[3]:off[3] + n_tok], ints[off[4]:off[4] + n_tok]
            lens = ints[off[5]:off[5] + B]
            assert np.array_equal(lens, s.lens[t])
            act = np.nonzero(s.lens[t] > 0)[0]
            assert np.array_equal(tseq, act) and np.array_equal(tpos, s.lens[t, act] - 1)
            assert np.array_equal(rows[r1:r1 + n_tok], W.token_row(s.resp[t, act], s.lens[t, act] - 1))
            for sl, r_, n_ in s.prefill[t]:
                sel = pseq == sl
                assert np.array_equal(ppos[sel], np.arange(n_)) and plens[sl] == n_
                assert np.array_equal(rows[r0:r0 + n_pre][sel], W.token_row(r_, np.arange(n_)))
            assert np.all((ppos < plens[pseq]) if n_pre else True)
            assert np.all(tseq < B) and np.all(pseq < B)
