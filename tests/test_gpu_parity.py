"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Packed codes, scales and offsets must match bit for bit;
bf16 attention outputs within max-abs 2e-3 / mean-abs 2e-4 of the fp64 oracle.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from kv4_case import Case, compare_outputs  # noqa: E402
from int8_kv_cache_kv4_gb300 import kv4  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kv4.load(build_if_missing=True)


# every decode kernel (work-balanced stream, warp-level mma split kernel,
# CUDA cores) must meet the bar; shapes a kernel does not support run the
# CUDA-core kernel, and the stream kernel runs the mma split kernel when
# max_splits > 0
@pytest.fixture(autouse=True, params=[kv4.KV4_KERNEL_STREAM, kv4.KV4_KERNEL_MMA_SYNC,
                                      kv4.KV4_KERNEL_CUDA_CORE],
                ids=["stream", "mma", "cuda"])
def kernel(request):
    prev = kv4.kv4_set_decode_kernel(request.param)
    yield request.param
    kv4.kv4_set_decode_kernel(prev)


def _bytes_equal(gpu_t, ref, what):
    got = gpu_t.cpu().numpy()[: ref.size]
    if not np.array_equal(got, ref):
        bad = np.nonzero(got != ref)[0]
        raise AssertionError(f"{what}: {bad.size} bytes differ, first at {bad[:8]}")


# ------------------------------------------------------------ tiny config
def test_tiny_config_append_bit_exact_and_decode():
    # 4 sequences x 512, S=4, R=64, group 32: a 511-token populate append,
    # a one-token append, then decode (seed 1)
    c = Case([512] * 4, S=4, R=64, g=32, seed=1, extra_pages=128 - 4 * 32)
    assert c.num_pages == 128
    g = c.gpu()
    paged, side, st = c.oracle_cache()
    assert st == 0 and g.read_status() == 0
    _bytes_equal(g.paged, paged, "paged INT4 cache")
    _bytes_equal(g.side, side, "INT8 side cache")
    out, lse = c.gpu_decode(g)
    ref, rlse = c.oracle_decode()
    mx, mean = compare_outputs(out, lse, ref, rlse, range(c.B), c.lens)
    print(f"tiny: max abs {mx:.2e} mean abs {mean:.2e}")


@pytest.mark.parametrize("g_", [32, 64, 128])
@pytest.mark.parametrize("S,R", [(4, 64), (0, 0), (4, 0), (0, 16), (16, 128)])
def test_append_bit_exact_groups_and_windows(g_, S, R):
    c = Case([200, 37, 1, 64], S=S, R=R, g=g_, seed=5, h_q=8, h_kv=2)
    gc = c.gpu()
    paged, side, st = c.oracle_cache()
    assert st == 0 and gc.read_status() == 0
    _bytes_equal(gc.paged, paged, "paged INT4 cache")
    _bytes_equal(gc.side, side, "INT8 side cache")
    out, lse = c.gpu_decode(gc)
    ref, rlse = c.oracle_decode()
    compare_outputs(out, lse, ref, rlse, range(c.B), c.lens)


@pytest.mark.parametrize("h_q,h_kv,d_h", [(32, 8, 128), (8, 8, 128), (16, 2, 128), (16, 4, 64)])
def test_decode_ragged_lengths_and_splits(h_q, h_kv, d_h):
    # L = 0, 1, below S, exactly S, mid-page, page-aligned, S+R-crossing, long
    lens = [0, 1, 3, 4, 17, 64, 84, 85, 700, 1500]
    c = Case(lens, S=4, R=80, g=32, seed=6, h_q=h_q, h_kv=h_kv, d_h=d_h)
    gc = c.gpu()
    ref, rlse = c.oracle_decode()
    for ms in (0, 1, 3, 17):
        out, lse = c.gpu_decode(gc, max_splits=ms)
        compare_outputs(out, lse, ref, rlse, range(c.B), c.lens)


def test_all_int8_when_window_covers_sequence():
    c = Case([300, 513, 20], S=4, R=1024, g=32, seed=7, h_q=16, h_kv=4)
    gc = c.gpu()
    paged, side, _ = c.oracle_cache()
    _bytes_equal(gc.side, side, "INT8 side cache")
    out, lse = c.gpu_decode(gc)
    ref, rlse = c.oracle_decode()
    compare_outputs(out, lse, ref, rlse, range(c.B), c.lens)


def test_bf16_comparator_matches_unquantized_attention():
    c = Case([1, 33, 400, 1000], S=4, R=64, g=32, seed=8, h_q=16, h_kv=4)
    gc = c.gpu(with_bf16=True)
    out, lse = c.gpu_decode(gc, bf16=True)
    ref, rlse = c.oracle_bf16()
    compare_outputs(out, lse, ref, rlse, range(c.B), c.lens)


@pytest.mark.parametrize("max_splits", [0, 3])
def test_bf16_comparator_tensor_core_kernel(max_splits):
    # head_dim 128, 4 query heads per kv head: with max_splits = 0 the
    # tensor-core kernel (64-page work items claimed by warps; lengths with
    # partial pages, several items per pair, an empty and a one-token
    # sequence), else the split kernel; both against exact attention, and the
    # tensor-core result repeated bit for bit
    c = Case([0, 1, 15, 16, 17, 511, 512, 513, 1100, 5000], S=4, R=64, g=32, seed=12)
    gc = c.gpu(with_bf16=True)
    out, lse = c.gpu_decode(gc, max_splits=max_splits, bf16=True)
    ref, rlse = c.oracle_bf16()
    compare_outputs(out, lse, ref, rlse, range(c.B), c.lens)
    out2, lse2 = c.gpu_decode(gc, max_splits=max_splits, bf16=True)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    assert gc.read_status() == 0


def test_split_combine_against_oracle():
    rng = np.random.default_rng(9)
    rows, n, d = 37, 11, 128
    po = rng.standard_normal((rows, n, d)).astype(np.float32)
    pl = (rng.standard_normal((rows, n)) * 3).astype(np.float32)
    pl[rng.random((rows, n)) < 0.3] = -np.inf
    pl[5, :] = -np.inf  # an all-empty row
    out = torch.empty((rows, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((rows,), dtype=torch.float32, device="cuda")
    kv4.kv4_split_combine(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), out, lse)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    z = lse.cpu().numpy()
    for r in range(rows):
        ro, rz = oracle.combine(po[r].astype(np.float64), pl[r].astype(np.float64))
        if rz == -np.inf:
            assert np.all(o[r] == 0) and z[r] == -np.inf
            continue
        assert np.max(np.abs(o[r] - ro)) <= 2e-3 + 4e-3 * np.max(np.abs(ro))
        assert abs(z[r] - rz) <= 1e-5 * max(1.0, abs(rz))


def test_bad_block_table_entries_set_status_without_fault():
    c = Case([100, 60], S=4, R=16, g=32, seed=10, h_q=8, h_kv=2)
    gc = c.gpu()
    gc.clear_status()
    bt = c.bt.copy()
    bt[0, 2] = c.num_pages + 5   # beyond the pool
    bt[1, 1] = -7
    gc.set_block_table(bt)
    out, lse = c.gpu_decode(gc)
    assert gc.read_status() & kv4.KV4_STATUS_BAD_PAGE
    assert np.all(np.isfinite(out))
    # appends through a bad entry are skipped and reported, not faulted
    gc.clear_status()
    k, v, s, p, la = c.tokens(1)
    dev = torch.device("cuda")
    bt2 = c.bt.copy()
    bt2[0, (int(c.lens[0]) - 1) // 16] = 10 ** 6
    gc.set_block_table(bt2)
    before = gc.paged.clone()
    gc.append(torch.from_numpy(k.view(np.int16)).to(dev).view(torch.bfloat16)[:1],
              torch.from_numpy(v.view(np.int16)).to(dev).view(torch.bfloat16)[:1],
              torch.from_numpy(s[:1]).to(dev), torch.from_numpy(p[:1]).to(dev),
              torch.from_numpy(la).to(dev))
    torch.cuda.synchronize()
    assert gc.read_status() & kv4.KV4_STATUS_BAD_PAGE
    assert torch.equal(before, gc.paged)


def test_host_argument_errors_enqueue_nothing():
    c = Case([16], S=4, R=16, g=32, seed=11, h_q=8, h_kv=2)
    gc = c.gpu()
    bad = kv4.make_layout(h_q=8, h_kv=2, d_h=96, group=32, sink=4, recent=16, max_seqs=1,
                          num_pages=c.num_pages, max_pages_per_seq=c.mpps)
    with pytest.raises(kv4.KV4Error):
        kv4.kv4_quant_append(bad, gc.paged, gc.side,
                             torch.zeros((1, 2, 128), dtype=torch.bfloat16, device="cuda"),
                             torch.zeros((1, 2, 128), dtype=torch.bfloat16, device="cuda"),
                             torch.zeros(1, dtype=torch.int32, device="cuda"),
                             torch.zeros(1, dtype=torch.int32, device="cuda"),
                             torch.ones(1, dtype=torch.int32, device="cuda"), gc.block_table)
    q = torch.zeros((1, 8, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    small_ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(kv4.KV4Error, match="workspace"):
        kv4.kv4_decode_attn(gc.layout, gc.paged, gc.side, q, torch.ones(1, dtype=torch.int32,
                            device="cuda"), gc.block_table, small_ws, out)


def test_sequence_filling_its_block_table_row():
    # L = max_pages_per_seq * 16: the last page is full and the row has no spare entry
    c = Case([256, 240, 17], S=4, R=32, g=32, seed=12, h_q=8, h_kv=2)
    assert c.mpps * 16 == 256
    gc = c.gpu()
    out, lse = c.gpu_decode(gc)
    assert gc.read_status() == 0
    ref, rlse = c.oracle_decode()
    compare_outputs(out, lse, ref, rlse, range(c.B), c.lens)


def test_lengths_outside_the_block_table_are_reported_and_read_as_empty():
    # a length past the row's capacity or negative: the kernels' own checks
    # report KV4_STATUS_BAD_LEN and treat the sequence as empty; the others
    # are unaffected
    c = Case([100, 60, 33], S=4, R=16, g=32, seed=13, h_q=8, h_kv=2)
    gc = c.gpu()
    gc.clear_status()
    lens = c.lens.copy()
    lens[1] = c.mpps * 16 + 1
    lens[2] = -5
    dev = torch.device("cuda")
    q = torch.from_numpy(c.q.view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty((c.B, c.h_q, c.d_h), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((c.B, c.h_q), dtype=torch.float32, device=dev)
    gc.decode(q, torch.from_numpy(lens).to(dev), out, lse)
    torch.cuda.synchronize()
    assert gc.read_status() & kv4.KV4_STATUS_BAD_LEN
    o = out.float().cpu().numpy().astype(np.float64)
    z = lse.cpu().numpy().astype(np.float64)
    assert np.all(o[1:] == 0) and np.all(np.isneginf(z[1:]))
    ref, rlse = c.oracle_decode([0])
    compare_outputs(o, z, ref, rlse, [0], c.lens)
