"""GPU parity of the FP4 probe formats (KV4-RL App. D.4, Fig. A4(c)): the
NVFP4 and MXFP4 append kernel writes the oracle's bytes bit for bit (codes,
block scales, global scale; with and without the K rotation), the
reconstruction into the bf16 comparator cache equals the oracle's bf16
operands exactly, and the probe's attention meets the output tolerance."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from kv4_case import Case, compare_outputs  # noqa: E402
from int8_kv_cache_kv4_gb300 import kv4  # noqa: E402
from int8_kv_cache_kv4_gb300 import workloads as W  # noqa: E402
from int8_kv_cache_kv4_gb300.cache import FP4ProbeCache  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kv4.load(build_if_missing=True)


def _gpu(c, fmt, rotate):
    dev = torch.device("cuda")
    fc = FP4ProbeCache(fmt=fmt, h_q=c.h_q, h_kv=c.h_kv, d_h=c.d_h, max_seqs=c.B,
                       num_pages=c.num_pages, max_pages_per_seq=c.mpps, device=dev,
                       hadamard_k=rotate)
    fc.set_block_table(c.bt)
    to = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev).view(dt)
    for stage in (0, 1):
        k, v, s, p, la = c.tokens(stage)
        if len(s):
            fc.append(to(k, torch.int16).view(torch.bfloat16), to(v, torch.int16).view(torch.bfloat16),
                      to(s, torch.int32), to(p, torch.int32), to(la, torch.int32))
    torch.cuda.synchronize()
    return fc


def _oracle_bytes(c, fmt, rotate):
    cache = np.zeros(c.num_pages * c.h_kv * 2 * 16 * oracle.fp4_row_bytes(c.d_h), np.uint8)
    st = 0
    for stage in (0, 1):
        k, v, s, p, la = c.tokens(stage)
        st |= oracle.fp4_append(h_kv=c.h_kv, d_h=c.d_h, fmt=fmt, rotate_k=rotate, max_seqs=c.B,
                                num_pages=c.num_pages, max_pages_per_seq=c.mpps, cache=cache,
                                k_new=k, v_new=v, tok_seq=s, tok_pos=p, seq_lens=la,
                                block_table=c.bt)
    return cache, st


@pytest.mark.parametrize("fmt", [kv4.KV4_FP4_NVFP4, kv4.KV4_FP4_MXFP4], ids=["nvfp4", "mxfp4"])
@pytest.mark.parametrize("rotate", [False, True], ids=["plain", "hadamard"])
@pytest.mark.parametrize("d_h", [128, 64])
def test_fp4_append_reconstruction_and_decode(fmt, rotate, d_h):
    c = Case([300, 37, 1, 160, 0], S=0, R=0, g=32, seed=40 + d_h, h_q=8, h_kv=2, d_h=d_h)
    fc = _gpu(c, fmt, rotate)
    ref, st = _oracle_bytes(c, fmt, rotate)
    assert st == 0 and fc.read_status() == 0
    got = fc.cache.cpu().numpy()
    if not np.array_equal(got, ref):
        bad = np.nonzero(got != ref)[0]
        raise AssertionError(f"{bad.size} probe-cache bytes differ, first at {bad[:8]}")
    # reconstruction: every written position equals the oracle's bf16 operand
    fc.reconstruct()
    torch.cuda.synchronize()
    bf = fc.bf16.cpu().numpy().view(np.uint16).reshape(c.num_pages, c.h_kv, 2, 16, d_h)
    for b in range(c.B):
        L = int(c.lens[b])
        if L == 0:
            continue
        kh, vh, _ = oracle.fp4_dequant_seq(c.k[b], c.v[b], fmt=fmt, rotate_k=rotate)
        pos = np.arange(L)
        pages = c.bt[b, pos // 16]
        for kv, want in ((0, kh), (1, vh)):
            rows = bf[pages, :, kv, pos % 16].transpose(1, 0, 2)      # [h_kv][L][d]
            assert np.array_equal(W.bf16_bits_to_f32(rows).astype(np.float64), want), (b, kv)
    # probe attention (bf16 operands) against the oracle's
    q = torch.from_numpy(c.q.view(np.int16)).cuda().view(torch.bfloat16)
    lens = torch.from_numpy(c.lens).cuda()
    out = torch.empty((c.B, c.h_q, d_h), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((c.B, c.h_q), dtype=torch.float32, device="cuda")
    fc.decode(q, lens, out, lse)
    torch.cuda.synchronize()
    ro, rl = {}, {}
    for b in range(c.B):
        qb = oracle.hadamard_bf16(c.q[b]) if rotate else c.q[b]
        ro[b], rl[b], _ = oracle.fp4_decode_seq(qb, c.k[b], c.v[b], fmt=fmt, sm_scale=c.sm_scale,
                                                rotate_k=rotate)
    compare_outputs(out.float().cpu().numpy().astype(np.float64),
                    lse.cpu().numpy().astype(np.float64), ro, rl, range(c.B), c.lens)


def test_fp4_nonfinite_vector_stored_as_zeros():
    c = Case([20], S=0, R=0, g=32, seed=50, h_q=8, h_kv=2)
    dev = torch.device("cuda")
    fc = FP4ProbeCache(fmt=kv4.KV4_FP4_NVFP4, h_q=8, h_kv=2, d_h=128, max_seqs=1,
                       num_pages=c.num_pages, max_pages_per_seq=c.mpps, device=dev)
    fc.set_block_table(c.bt)
    k = torch.ones((1, 2, 128), dtype=torch.bfloat16, device=dev)
    k[0, 1, 7] = float("inf")
    v = torch.ones((1, 2, 128), dtype=torch.bfloat16, device=dev)
    fc.cache.fill_(0x5A)
    fc.append(k, v, torch.zeros(1, dtype=torch.int32, device=dev),
              torch.zeros(1, dtype=torch.int32, device=dev),
              torch.full((1,), 20, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    assert fc.read_status() & kv4.KV4_STATUS_NONFINITE
    rb = oracle.fp4_row_bytes(128)
    rows = fc.cache.cpu().numpy().reshape(c.num_pages, 2, 2, 16, rb)[c.bt[0, 0], :, :, 0]
    assert np.all(rows[1, 0, :64 + 8] == 0) and np.all(rows[1, 0, 64 + 12:] == 0)   # K of head 1
    assert np.any(rows[0, 0, :64] != 0x5A)                                         # head 0 written
