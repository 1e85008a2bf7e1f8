"""Closed forms of scheduling-induced KV concentration (KV4-RL Sec. 4.1,
Proposition 4.1, and App. C: renewal-reward analysis of continuous refill and
synchronous waves).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
report may import this module; the product path never does.  Plain numpy in
fp64, written from the definitions, over an explicit response-length pmf
(positive integer support).  Time is counted in decode steps; a response with
prompt length P and generation length L visits cached contexts P, P+1, ...,
P+L-1 (App. C.2), so its logical KV work is Q(P, L) = P L + L (L - 1) / 2.

Every function here is pinned in tests/test_oracle_concentration.py against
brute-force enumeration, hand-computed cases and the pages' own identities.
"""
from __future__ import annotations

import numpy as np


def _check(support, pmf):
    s = np.asarray(support, dtype=np.float64)
    p = np.asarray(pmf, dtype=np.float64)
    assert s.ndim == 1 and s.shape == p.shape and np.all(s >= 1) and np.all(p >= 0)
    assert np.all(np.diff(s) > 0), "support must be increasing"
    assert abs(p.sum() - 1.0) < 1e-9, "pmf must sum to 1"
    return s, p


def moments(support, pmf):
    """E[L] and E[L (L - 1)]."""
    s, p = _check(support, pmf)
    return float((s * p).sum()), float((s * (s - 1) * p).sum())


def max_moments(support, pmf, B: int):
    """E[M_B] and E[M_B^2] for M_B the maximum of B i.i.d. lengths.
    From the distribution of the maximum: Pr(M_B <= l) = F(l)^B, so
    Pr(M_B = l_k) = F(l_k)^B - F(l_(k-1))^B on the support points."""
    s, p = _check(support, pmf)
    F = np.minimum(np.cumsum(p), 1.0)
    Fb = F ** B
    pm = np.diff(np.concatenate([[0.0], Fb]))
    return float((s * pm).sum()), float((s * s * pm).sum())


def logical_work(P: float, support, pmf):
    """q = E[Q(P, L)] = P E[L] + E[L (L - 1)] / 2   (App. C.2)."""
    mu, m2 = moments(support, pmf)
    return P * mu + m2 / 2.0


def refill_mean_context(P: float, support, pmf):
    """Continuous refill: l_async = q / E[L] = P + E[L(L-1)] / (2 E[L])
    (Prop. 4.1; App. C eq. A4)."""
    mu, m2 = moments(support, pmf)
    return P + m2 / (2.0 * mu)


def refill_volume(P: float, support, pmf, B: int, kappa: float = 1.0):
    """Continuous refill: V_async = kappa B q / E[L]   (eq. A4)."""
    mu, _ = moments(support, pmf)
    return kappa * B * logical_work(P, support, pmf) / mu


def wave_volume(P: float, support, pmf, B: int, kappa: float = 1.0):
    """Synchronous waves: V_sync = kappa B q / E[M_B]   (eq. A6)."""
    em, _ = max_moments(support, pmf, B)
    return kappa * B * logical_work(P, support, pmf) / em


def wave_occupancy(support, pmf, B: int):
    """Synchronous waves: step-averaged active batch B E[L] / E[M_B]   (eq. A7)."""
    mu, _ = moments(support, pmf)
    em, _ = max_moments(support, pmf, B)
    return B * mu / em


def wave_mean_context(P: float, support, pmf, B: int):
    """Synchronous waves: step-averaged mean context of the active slots,
    P + (E[M_B^2] - E[M_B]) / (2 E[M_B])   (App. C.3)."""
    em, em2 = max_moments(support, pmf, B)
    return P + (em2 - em) / (2.0 * em)


def concentration(support, pmf, B: int):
    """C_KV = V_async / V_sync = E[M_B] / E[L]   (Prop. 4.1; eq. A8)."""
    mu, _ = moments(support, pmf)
    em, _ = max_moments(support, pmf, B)
    return em / mu


def length_biased(support, pmf):
    """Length seen at a decode step under continuous refill:
    Pr(L* = l) = l Pr(L = l) / E[L]; the age is then uniform on 0..l-1 (eq. A5)."""
    s, p = _check(support, pmf)
    q = s * p
    return q / q.sum()
