"""GPU run of the KV-concentration driver: continuous-refill and
synchronous-wave schedules (KV4-RL Prop. 4.1) driven through the C ABI, with
slots refilled by new responses mid-run.  At the last step every active
slot's decode output matches the oracle on that slot's regenerated response,
and no status bit is raised."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from kv4_case import compare_outputs  # noqa: E402
from int8_kv_cache_kv4_gb300 import kv4, rollout as R, workloads as W  # noqa: E402

SHAPE = dict(h_q=16, h_kv=4, d_h=128, group=32, sink=4, recent=16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kv4.load(build_if_missing=True)


def _check_last_step(sched, res, seed, rotate_k=False):
    t = sched.steps - 1
    out = res["out"].float().numpy().astype(np.float64)
    lse = res["lse"].numpy().astype(np.float64)
    act = np.nonzero(sched.lens[t] > 0)[0]
    assert len(act) > 0
    ref_o, ref_l = {}, {}
    for b in act:
        k, v, q = R.slot_sources(sched, t, int(b), h_q=SHAPE["h_q"], h_kv=SHAPE["h_kv"],
                                 d_h=SHAPE["d_h"], seed=seed)
        if rotate_k:
            q = oracle.hadamard_bf16(q)
        ref_o[b], ref_l[b], st = oracle.decode_seq(q, k, v, g=SHAPE["group"], S=SHAPE["sink"],
                                                   R=SHAPE["recent"], sm_scale=1 / math.sqrt(128),
                                                   rotate_k=rotate_k)
        assert st == 0
    compare_outputs(out, lse, ref_o, ref_l, act, sched.lens[t])
    idle = np.nonzero(sched.lens[t] == 0)[0]
    assert np.all(out[idle] == 0)


@pytest.mark.parametrize("rotate_k", [False, True], ids=["plain", "hadamard"])
def test_refill_schedule_parity(rotate_k):
    sup, pmf = W.lognormal_length_pmf(50, 0.8, 5, 400)
    s = R.refill_schedule(12, 20, sup, pmf, 160, np.random.default_rng(31))
    assert sum(len(p) for p in s.prefill[1:]) > 5          # responses were replaced mid-run
    res = R.drive(s, seed=31, chunk=16, hadamard_k=rotate_k, **SHAPE)
    assert res["status"] == 0
    _check_last_step(s, res, 31, rotate_k)
    assert np.all(res["decode_ms"] > 0)


def test_wave_schedule_parity():
    sup, pmf = W.lognormal_length_pmf(50, 0.8, 5, 400)
    s = R.wave_schedule(12, 20, sup, pmf, 2, np.random.default_rng(32))
    # cut inside the second wave, while some slots are idle and some still run
    w0 = next(t for t in range(1, s.steps) if len(s.prefill[t]))
    cut = w0 + int(np.sort((s.lens[w0:] > 0).sum(axis=0))[len(s.lens[0]) // 2])
    s = R.Schedule(s.kind, s.B, s.P, s.lens[:cut], s.resp[:cut], s.prefill[:cut])
    assert (s.lens[-1] == 0).any() and (s.lens[-1] > 0).any()
    res = R.drive(s, seed=32, chunk=16, **SHAPE)
    assert res["status"] == 0
    _check_last_step(s, res, 32)
