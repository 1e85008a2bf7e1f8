"""Pins for the oracle's KV-concentration closed forms (KV4-RL Prop. 4.1 and
App. C eqs. A4-A8): brute-force enumeration of the wave maximum, hand-worked
cases, the pages' own identities (the variance form of eq. A4, the mean age
under eq. A5), limits (B = 1, degenerate lengths), and direct step-by-step
simulation with plain loops.  A dropped term in q, the wrong power of F in
the maximum's distribution, or a missing 1/2 fails at least one of them.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import concentration as C
from int8_kv_cache_kv4_gb300 import workloads as W

SUP = np.array([1, 2, 5])
PMF = np.array([0.2, 0.5, 0.3])


@pytest.mark.parametrize("B", [1, 2, 3, 4])
def test_wave_maximum_against_enumeration(B):
    em = em2 = 0.0
    for tup in itertools.product(range(3), repeat=B):
        pr = math.prod(PMF[i] for i in tup)
        m = max(SUP[i] for i in tup)
        em += pr * m
        em2 += pr * m * m
    got = C.max_moments(SUP, PMF, B)
    assert got[0] == pytest.approx(em, abs=1e-12) and got[1] == pytest.approx(em2, abs=1e-12)


def test_two_point_case_by_hand():
    # L in {1, 3} with equal probability, B = 2: M_2 = 3 unless both are 1
    sup, pmf, P = np.array([1, 3]), np.array([0.5, 0.5]), 7
    assert C.moments(sup, pmf) == (2.0, 3.0)              # E[L], E[L(L-1)] = (0 + 6) / 2
    assert C.max_moments(sup, pmf, 2) == (2.5, 7.0)       # 1/4 * 1 + 3/4 * 3;  1/4 + 3/4 * 9
    assert C.concentration(sup, pmf, 2) == 1.25
    assert C.refill_mean_context(P, sup, pmf) == P + 0.75
    # waves: M = 1 (reward P, 1 step) w.p. 1/4, M = 3 (reward 3P + 3, 3 steps) w.p. 3/4
    assert C.wave_mean_context(P, sup, pmf, 2) == pytest.approx(
        float((Fraction(1, 4) * P + Fraction(3, 4) * (3 * P + 3)) / Fraction(5, 2)), abs=1e-12)
    q = P * 2 + 3 / 2
    assert C.logical_work(P, sup, pmf) == q
    assert C.refill_volume(P, sup, pmf, 2, kappa=3.0) == pytest.approx(3 * 2 * q / 2)
    assert C.wave_volume(P, sup, pmf, 2, kappa=3.0) == pytest.approx(3 * 2 * q / 2.5)
    assert C.wave_occupancy(sup, pmf, 2) == pytest.approx(2 * 2 / 2.5)


def test_degenerate_lengths_and_single_slot():
    sup, pmf = np.array([40]), np.array([1.0])
    for B in (1, 2, 64):
        assert C.concentration(sup, pmf, B) == 1.0
        assert C.wave_occupancy(sup, pmf, B) == B
        assert C.wave_mean_context(10, sup, pmf, B) == pytest.approx(10 + 39 / 2)
    assert C.refill_mean_context(10, sup, pmf) == pytest.approx(10 + 39 / 2)
    # B = 1: the wave is one response, so both schedules coincide
    assert C.concentration(SUP, PMF, 1) == pytest.approx(1.0)
    assert C.wave_volume(3, SUP, PMF, 1) == pytest.approx(C.refill_volume(3, SUP, PMF, 1))


def test_concentration_exceeds_one_and_grows_with_batch():
    # Prop. 4.1: C_KV > 1 for a non-degenerate distribution and B >= 2
    sup, pmf = W.lognormal_length_pmf(3000, 0.8, 256, 16384)
    prev = 1.0
    for B in (2, 4, 16, 64, 256):
        c = C.concentration(sup, pmf, B)
        assert c > prev
        prev = c
    assert prev < sup.max() / C.moments(sup, pmf)[0] + 1e-9   # M_B <= max length


def test_variance_form_and_mean_age():
    # eq. A4 in the pages' variance form: P + (mu - 1)/2 + sigma^2 / (2 mu)
    sup, pmf = W.lognormal_length_pmf(300, 0.6, 16, 2000)
    mu = float((sup * pmf).sum())
    var = float((sup * sup * pmf).sum()) - mu * mu
    assert C.refill_mean_context(5, sup, pmf) == pytest.approx(5 + (mu - 1) / 2 + var / (2 * mu),
                                                               rel=1e-12)
    # eq. A5: the length-biased pmf sums to one and its mean age is E[L(L-1)] / (2 mu)
    lb = C.length_biased(sup, pmf)
    assert lb.sum() == pytest.approx(1.0, abs=1e-12)
    age = float((lb * (sup - 1) / 2).sum())
    assert age == pytest.approx(C.moments(sup, pmf)[1] / (2 * mu), rel=1e-12)


def _simulate(sup, pmf, B, P, steps, rng, waves):
    """Plain step-by-step simulation: returns the step averages of the
    resident context sum, of the active count and of the mean active context."""
    vol = act = ctx = 0.0
    if not waves:
        rem = [0] * B
        age = [0] * B
        for _ in range(steps):
            s_v = 0
            for i in range(B):
                if rem[i] == 0:     # refilled before this step
                    rem[i] = int(rng.choice(sup, p=pmf))
                    age[i] = 0
                s_v += P + age[i]
                age[i] += 1
                rem[i] -= 1
            vol += s_v
            act += B
            ctx += s_v / B
        return vol / steps, act / steps, ctx / steps
    n = 0
    while n < steps:
        L = [int(x) for x in rng.choice(sup, p=pmf, size=B)]
        for t in range(max(L)):
            live = [i for i in range(B) if t < L[i]]
            vol += sum(P + t for _ in live)
            act += len(live)
            ctx += P + t
            n += 1
    return vol / n, act / n, ctx / n


def test_direct_simulation_matches_closed_forms():
    sup, pmf, B, P = np.array([1, 2, 3, 8]), np.array([0.4, 0.3, 0.2, 0.1]), 4, 5
    rng = np.random.default_rng(11)
    v_r, a_r, c_r = _simulate(sup, pmf, B, P, 60000, rng, waves=False)
    v_w, a_w, c_w = _simulate(sup, pmf, B, P, 60000, rng, waves=True)
    assert v_r == pytest.approx(C.refill_volume(P, sup, pmf, B), rel=0.02)
    assert c_r == pytest.approx(C.refill_mean_context(P, sup, pmf), rel=0.02)
    assert v_w == pytest.approx(C.wave_volume(P, sup, pmf, B), rel=0.02)
    assert a_w == pytest.approx(C.wave_occupancy(sup, pmf, B), rel=0.02)
    assert c_w == pytest.approx(C.wave_mean_context(P, sup, pmf, B), rel=0.02)
    assert v_r / v_w == pytest.approx(C.concentration(sup, pmf, B), rel=0.03)


def test_lognormal_pmf_matches_its_sampler():
    # the input recipe's lognormal lengths and their pmf agree (chi-square-like)
    sup, pmf = W.lognormal_length_pmf(3000, 0.8, 256, 16384)
    rng = np.random.default_rng(5)
    x = np.clip(np.round(np.exp(rng.normal(math.log(3000), 0.8, size=400000))), 256, 16384)
    edges = np.unique(np.floor(np.quantile(x, np.linspace(0, 1, 21))) + 0.5)  # between integers
    edges[0], edges[-1] = 255.5, 16384.5
    counts, _ = np.histogram(x, bins=edges)
    cdf = np.concatenate([[0.0], np.cumsum(pmf)])
    idx = np.searchsorted(sup, edges, side="right")
    expect = np.diff(cdf[np.clip(idx, 0, len(sup))]) * len(x)
    assert np.all(np.abs(counts - expect) <= 5 * np.sqrt(expect) + 1)
