"""GPU parity of the work-balanced decode kernel's scheduling: the stream of
16-slot protected units and two-page INT4 units cut into CTA shares of equal
cost and walked by the warps of each CTA.
Cases aim at the bookkeeping -- pairs spread over many CTAs, CTAs without
work, empty and very short sequences, partly filled recent-window rings,
more sequences than threads in the start search -- and compare with the
CPU oracle like the other parity tests."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from kv4_case import Case, compare_outputs  # noqa: E402
from int8_kv_cache_kv4_gb300 import kv4  # noqa: E402


@pytest.fixture(scope="module", autouse=True, params=[kv4.KV4_KERNEL_STREAM], ids=["stream"])
def _lib(request):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kv4.load(build_if_missing=True)
    prev = kv4.kv4_set_decode_kernel(request.param)
    yield
    kv4.kv4_set_decode_kernel(prev)


def _run(c):
    gc = c.gpu()
    gc.clear_status()
    out, lse = c.gpu_decode(gc)
    assert gc.read_status() == 0
    ref, rlse = c.oracle_decode()
    return compare_outputs(out, lse, ref, rlse, range(c.B), c.lens)


def test_one_long_sequence_spread_over_many_ctas():
    # 8 pairs of ~1250 pages each: every pair's INT4 region spans ~90 CTAs
    _run(Case([20000], S=4, R=128, g=32, seed=21))


def test_single_token_leaves_most_ctas_without_work():
    _run(Case([1], S=4, R=64, g=32, seed=22))


def test_all_sequences_empty():
    _run(Case([0, 0, 0], S=4, R=64, g=32, seed=23, h_q=8, h_kv=2))


@pytest.mark.parametrize("g_", [32, 64, 128])
def test_many_short_sequences_and_partial_rings(g_):
    # 300 sequences (more than the 128 threads of the start search): empty,
    # shorter than the sinks, inside the ring (S < L <= S + R), page-aligned
    # and longer, in seeded order
    rng = np.random.default_rng(24)
    kinds = [0, 1, 3, 4, 5, 17, 36, 68, 69, 70, 80, 96, 128, 200, 333, 511, 512]
    lens = list(rng.choice(kinds, size=300))
    _run(Case(lens, S=4, R=64, g=g_, seed=25, h_q=8, h_kv=2))


@pytest.mark.parametrize("S,R", [(0, 0), (4, 0), (0, 16), (3, 13), (16, 128)])
def test_window_shapes(S, R):
    # sink / window sizes that are not multiples of the 8-slot unit
    _run(Case([1, 2, 3, 15, 16, 17, 29, 150, 777], S=S, R=R, g=32, seed=26, h_q=16, h_kv=4))


@pytest.mark.parametrize("where", ["spread", "front"])
def test_few_long_sequences_among_idle_slots(where):
    # a batch of 240 slots with four long sequences (a synchronous wave's
    # tail): interleaved with idle slots, or all in front of a tail of idle ones
    lens = np.zeros(240, dtype=np.int64)
    pos = [3, 77, 150, 239] if where == "spread" else [0, 1, 2, 3]
    lens[pos] = [2500, 3100, 1800, 2900]
    c = Case(lens, S=4, R=64, g=32, seed=24, h_q=8, h_kv=2)
    _run(c)


@pytest.mark.parametrize("B", [12, 4], ids=["tickets", "merge-kernel"])
def test_back_to_back_calls_on_one_workspace(B):
    # Calls enqueued back to back on one stream and sharing one workspace: each
    # decode call's prep kernel rewrites the plan while the decode before it
    # finishes, and zeroes the tickets once it has; an append between calls
    # starts during the previous decode's tail.  Every output must equal, bit
    # for bit, that of the same call made alone.  B = 12 (96 pairs) merges in
    # the decode kernel, B = 4 (32 pairs) in the separate merge kernel.
    rng = np.random.default_rng(40 + B)
    mixes = [list(rng.integers(0, 6000, B)), [20000] + [0] * (B - 1), list(rng.integers(1, 300, B))]
    cases = [Case(m, S=4, R=128, g=32, seed=41 + i) for i, m in enumerate(mixes)]
    gcs = [c.gpu() for c in cases]
    alone = [c.gpu_decode(gc) for c, gc in zip(cases, gcs)]
    # one workspace, as large as the largest of the three calls needs
    nbytes = max(kv4.workspace_bytes(gc.layout, B, 0) for gc in gcs)
    shared = torch.empty(nbytes, dtype=torch.uint8, device=gcs[0].device)
    for gc in gcs:
        gc._ws[(B, 0, False)] = shared
    dev = gcs[0].device
    order = [0, 1, 2, 1, 0, 2, 2, 0]
    ins = [(torch.from_numpy(c.q.view(np.int16)).to(dev).view(torch.bfloat16),
            torch.from_numpy(c.lens).to(dev)) for c in cases]
    outs = [(torch.empty((B, cases[i].h_q, cases[i].d_h), dtype=torch.bfloat16, device=dev),
             torch.empty((B, cases[i].h_q), dtype=torch.float32, device=dev)) for i in order]
    k, v, s, p, la = cases[0].tokens(1)
    to = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev).view(dt)  # noqa: E731
    app = (to(k, torch.int16).view(torch.bfloat16), to(v, torch.int16).view(torch.bfloat16),
           to(s, torch.int32), to(p, torch.int32), to(la, torch.int32))
    torch.cuda.synchronize()
    for n, i in enumerate(order):
        if n == 4 and len(s):
            gcs[0].append(*app)  # rewrites case 0's step token with the same bytes
        gcs[i].decode(ins[i][0], ins[i][1], outs[n][0], outs[n][1])
    torch.cuda.synchronize()
    for gc in gcs:
        assert gc.read_status() == 0
    for n, i in enumerate(order):
        assert np.array_equal(outs[n][0].float().cpu().numpy(), alone[i][0].astype(np.float32)), (n, i)
        assert np.array_equal(outs[n][1].cpu().numpy(), alone[i][1].astype(np.float32)), (n, i)
