"""GPU parity of the Hadamard K-rotation (KV4-RL Sec. 3 eq. 3.4; App. A.3
"Encoding and allocation"; App. D.4 K-only): the query rotation and the
rotating append are bit-exact against the CPU oracle, and decode over a
rotated cache with rotated queries meets the same output tolerance as the
unrotated path, for every decode kernel.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from kv4_case import Case, compare_outputs  # noqa: E402
from int8_kv_cache_kv4_gb300 import kv4  # noqa: E402
from int8_kv_cache_kv4_gb300 import workloads as W  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kv4.load(build_if_missing=True)


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _bytes_equal(gpu_t, ref, what):
    got = gpu_t.cpu().numpy()[: ref.size]
    if not np.array_equal(got, ref):
        bad = np.nonzero(got != ref)[0]
        raise AssertionError(f"{what}: {bad.size} bytes differ, first at {bad[:8]}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("rows", [1, 7, 8, 9, 1000, 4099])
def test_query_rotation_bit_exact(d, rows):
    rng = np.random.default_rng(rows * 3 + d)
    x = (rng.standard_normal((rows, d)) * np.exp2(rng.integers(-6, 7, size=(rows, 1))))
    x[:, rng.integers(0, d)] *= 40.0                 # an outlier channel
    x[0, :] = 0.0 if rows > 1 else x[0, :]           # an all-zero row
    bits = W.f32_to_bf16_bits(x.astype(np.float32))
    ref = oracle.hadamard_bf16(bits)
    xd = _bf16_dev(bits)
    y = torch.empty_like(xd)
    kv4.kv4_hadamard_bf16(xd, y)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y), ref)
    assert np.array_equal(_bits(xd), bits)           # input untouched
    kv4.kv4_hadamard_bf16(xd)                        # in place
    torch.cuda.synchronize()
    assert np.array_equal(_bits(xd), ref)


def test_query_rotation_of_decode_shaped_query():
    q = W.q_numpy(77, 64, 32, 128)                   # [B][h_q][d_h]
    qd = _bf16_dev(q)
    out = kv4.kv4_hadamard_bf16(qd, torch.empty_like(qd))
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), oracle.hadamard_bf16(q))


@pytest.mark.parametrize("g_", [32, 64, 128])
@pytest.mark.parametrize("S,R", [(4, 64), (0, 0), (16, 128)])
def test_rotated_append_bit_exact_and_decode(g_, S, R):
    c = Case([200, 37, 1, 64, 0], S=S, R=R, g=g_, seed=15, h_q=8, h_kv=2, rotate_k=True)
    gc = c.gpu()
    paged, side, st = c.oracle_cache()
    assert st == 0 and gc.read_status() == 0
    _bytes_equal(gc.paged, paged, "paged INT4 cache (rotated K)")
    _bytes_equal(gc.side, side, "INT8 side cache (rotated K)")
    out, lse = c.gpu_decode(gc)
    ref, rlse = c.oracle_decode()
    compare_outputs(out, lse, ref, rlse, range(c.B), c.lens)


def test_rotated_append_head_dim_64():
    c = Case([90, 300, 5], S=4, R=32, g=32, seed=16, h_q=16, h_kv=4, d_h=64, rotate_k=True)
    gc = c.gpu()
    paged, side, st = c.oracle_cache()
    assert st == 0
    _bytes_equal(gc.paged, paged, "paged INT4 cache (rotated K, d_h 64)")
    _bytes_equal(gc.side, side, "INT8 side cache (rotated K, d_h 64)")
    out, lse = c.gpu_decode(gc)
    ref, rlse = c.oracle_decode()
    compare_outputs(out, lse, ref, rlse, range(c.B), c.lens)


@pytest.mark.parametrize("which", [kv4.KV4_KERNEL_STREAM, kv4.KV4_KERNEL_MMA_SYNC,
                                   kv4.KV4_KERNEL_CUDA_CORE],
                         ids=["stream", "mma", "cuda"])
def test_rotated_decode_every_kernel(which):
    lens = [0, 1, 3, 4, 17, 64, 84, 85, 700, 1500]
    c = Case(lens, S=4, R=80, g=32, seed=17, h_q=32, h_kv=8, rotate_k=True)
    prev = kv4.kv4_set_decode_kernel(which)
    try:
        gc = c.gpu()
        ref, rlse = c.oracle_decode()
        out, lse = c.gpu_decode(gc)
        compare_outputs(out, lse, ref, rlse, range(c.B), c.lens)
    finally:
        kv4.kv4_set_decode_kernel(prev)


def test_rotation_changes_only_k():
    # V bytes are identical with and without rotation; K bytes differ
    c0 = Case([100, 40], S=4, R=16, g=32, seed=18, h_q=8, h_kv=2)
    c1 = Case([100, 40], S=4, R=16, g=32, seed=18, h_q=8, h_kv=2, rotate_k=True)
    p0, p1 = c0.gpu().paged.cpu().numpy(), c1.gpu().paged.cpu().numpy()
    chunk = oracle.chunk_bytes(128, 32)
    half = 16 * 128 // 2
    a = p0.reshape(-1, chunk)
    b = p1.reshape(-1, chunk)
    assert np.array_equal(a[:, half:2 * half], b[:, half:2 * half])      # V codes
    assert not np.array_equal(a[:, :half], b[:, :half])                  # K codes


@pytest.mark.parametrize("which,splits", [(kv4.KV4_KERNEL_STREAM, 0), (kv4.KV4_KERNEL_MMA_SYNC, 0),
                                          (kv4.KV4_KERNEL_CUDA_CORE, 0), (kv4.KV4_KERNEL_AUTO, 3)],
                         ids=["stream", "mma", "cuda", "auto-splits3"])
def test_query_rotation_in_the_decode_call_equals_separate_rotation(which, splits):
    # kv4_decode_attn_hadamard (rotation inside the call: in the stream
    # kernel's query set-up, else into `out` first) against kv4_hadamard_bf16
    # followed by kv4_decode_attn: bit for bit, outputs and log-normalisers
    lens = [0, 1, 5, 64, 85, 333, 2100]
    c = Case(lens, S=4, R=80, g=32, seed=19, h_q=32, h_kv=8, rotate_k=True)
    prev = kv4.kv4_set_decode_kernel(which)
    try:
        gc = c.gpu()
        q = torch.from_numpy(c.q.view(np.int16)).cuda().view(torch.bfloat16)
        q0 = q.clone()
        lens_d = torch.from_numpy(c.lens).cuda()
        outs = []
        for sep in (False, True):
            out = torch.empty((c.B, c.h_q, c.d_h), dtype=torch.bfloat16, device="cuda")
            lse = torch.empty((c.B, c.h_q), dtype=torch.float32, device="cuda")
            gc.decode(q, lens_d, out, lse, max_splits=splits, separate_rotation=sep)
            torch.cuda.synchronize()
            outs.append((_bits(out), lse.cpu().numpy()))
        assert gc.read_status() == 0
        assert np.array_equal(_bits(q), _bits(q0))          # q untouched
        assert np.array_equal(outs[0][0], outs[1][0])
        assert np.array_equal(outs[0][1].view(np.uint32), outs[1][1].view(np.uint32))
    finally:
        kv4.kv4_set_decode_kernel(prev)
