"""CPU-side checks of the C ABI: the library builds for sm_103a, loads, exports
every entry point include/kv4.h declares, and its host-only functions
(validation, sizing, split plan) behave -- no GPU calls."""
import ctypes
import os
import subprocess

import pytest

from int8_kv_cache_kv4_gb300 import build, kv4


@pytest.fixture(scope="module")
def lib():
    build.build()
    return kv4.load()


def test_exports_every_declared_symbol(lib):
    names = kv4.declared_symbols()
    assert "kv4_quant_append" in names and "kv4_decode_attn" in names
    assert "kv4_split_combine" in names
    out = subprocess.run(["nm", "-D", "--defined-only", kv4.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing


def test_layout_validation(lib):
    ok = kv4.make_layout(max_seqs=4, num_pages=10, max_pages_per_seq=4)
    assert lib.kv4_check_layout(ctypes.byref(ok)) == kv4.KV4_OK
    for field, val, code in [("head_dim", 96, kv4.KV4_ERR_UNSUPPORTED),
                             ("page_size", 32, kv4.KV4_ERR_UNSUPPORTED),
                             ("int4_group", 16, kv4.KV4_ERR_UNSUPPORTED),
                             ("int8_group", 64, kv4.KV4_ERR_UNSUPPORTED),
                             ("num_q_heads", 12, kv4.KV4_ERR_INVALID_ARG),
                             ("sink", -1, kv4.KV4_ERR_INVALID_ARG),
                             ("num_pages", 0, kv4.KV4_ERR_INVALID_ARG)]:
        bad = kv4.make_layout(max_seqs=4, num_pages=10, max_pages_per_seq=4)
        setattr(bad, field, val)
        assert lib.kv4_check_layout(ctypes.byref(bad)) == code, field
        assert kv4.paged_cache_bytes(bad) == 0


def test_sizes_match_layout_description(lib):
    for g, chunk in [(32, 2560), (64, 2304), (128, 2176)]:
        lay = kv4.make_layout(group=g, max_seqs=3, num_pages=7, max_pages_per_seq=5)
        assert kv4.paged_cache_bytes(lay) == 7 * 8 * chunk
    lay = kv4.make_layout(sink=4, recent=128, max_seqs=3, num_pages=7, max_pages_per_seq=5)
    # per block: K8 and V8 codes 132 x 128 each, two scale arrays padded to 136
    assert kv4.side_cache_bytes(lay) == 3 * 8 * (2 * 132 * 128 + 4 * 136)
    lay = kv4.make_layout(sink=4, recent=124, max_seqs=3, num_pages=7, max_pages_per_seq=5)
    assert kv4.side_cache_bytes(lay) == 3 * 8 * (128 * 260)  # NS = 128: no padding
    assert kv4.bf16_cache_bytes(lay) == 7 * 8 * 2 * 16 * 128 * 2


def test_split_plan_and_workspace(lib):
    lay = kv4.make_layout(recent=256, max_seqs=1, num_pages=8192, max_pages_per_seq=8192)
    n = kv4.num_splits(lay, 1)
    assert n * 8 >= 2 * 152      # a single long request still fills the GPU
    assert kv4.workspace_bytes(lay, 1) >= 32 * n * (128 + 1) * 4
    lay = kv4.make_layout(max_seqs=64, num_pages=40000, max_pages_per_seq=512)
    assert kv4.num_splits(lay, 64, max_splits=1) == 2   # one INT4 split + one protected split
    assert kv4.workspace_bytes(lay, 0) == 0 or kv4.workspace_bytes(lay, 0) >= 0


def test_retired_kernel_ids_leave_the_selection_unchanged(lib):
    # only AUTO, CUDA_CORE, MMA_SYNC and STREAM select a kernel; other values
    # (3 and 5 named kernels that are no longer part of the library) are ignored
    prev = kv4.kv4_set_decode_kernel(kv4.KV4_KERNEL_STREAM)
    try:
        for bad in (3, 5, -1, 99):
            assert kv4.kv4_set_decode_kernel(bad) == kv4.KV4_KERNEL_STREAM
        assert kv4.kv4_set_decode_kernel(kv4.KV4_KERNEL_AUTO) == kv4.KV4_KERNEL_STREAM
    finally:
        kv4.kv4_set_decode_kernel(prev)


def test_null_arguments_rejected_on_host(lib):
    lay = kv4.make_layout(max_seqs=4, num_pages=10, max_pages_per_seq=4)
    rc = lib.kv4_quant_append(ctypes.byref(lay), None, None, None, None, None, None, 3, None,
                              None, None, None)
    assert rc == kv4.KV4_ERR_INVALID_ARG
    rc = lib.kv4_decode_attn(ctypes.byref(lay), None, None, None, None, 2, None, 0.1, 0, None, 0,
                             None, None, None, None)
    assert rc == kv4.KV4_ERR_INVALID_ARG
    assert lib.kv4_quant_append(ctypes.byref(lay), None, None, None, None, None, None, 0, None,
                                None, None, None) == kv4.KV4_OK   # T == 0: no-op
    assert lib.kv4_status_string(kv4.KV4_ERR_WORKSPACE) == b"workspace too small"


def test_hadamard_entry_points_validate_on_host(lib):
    # every rejection happens before any launch; rows == 0 / T == 0 are no-ops
    buf = ctypes.create_string_buffer(4096 + 16)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    assert lib.kv4_hadamard_bf16(base, base, 0, 128, None) == kv4.KV4_OK
    assert lib.kv4_hadamard_bf16(base, base, 4, 96, None) == kv4.KV4_ERR_INVALID_ARG
    assert lib.kv4_hadamard_bf16(base, base, -1, 128, None) == kv4.KV4_ERR_INVALID_ARG
    assert lib.kv4_hadamard_bf16(None, base, 4, 128, None) == kv4.KV4_ERR_INVALID_ARG
    assert lib.kv4_hadamard_bf16(base + 2, base + 2, 4, 64, None) == kv4.KV4_ERR_INVALID_ARG
    # y overlapping x without being x
    assert lib.kv4_hadamard_bf16(base, base + 8, 4, 128, None) == kv4.KV4_ERR_INVALID_ARG
    lay = kv4.make_layout(max_seqs=4, num_pages=10, max_pages_per_seq=4)
    rc = lib.kv4_quant_append_hadamard(ctypes.byref(lay), None, None, None, None, None, None, 3,
                                       None, None, None, None)
    assert rc == kv4.KV4_ERR_INVALID_ARG
    assert lib.kv4_quant_append_hadamard(ctypes.byref(lay), None, None, None, None, None, None,
                                         0, None, None, None, None) == kv4.KV4_OK
    rc = lib.kv4_decode_attn_hadamard(ctypes.byref(lay), None, None, None, None, 2, None, 0.1, 0,
                                      None, 0, None, None, None, None)
    assert rc == kv4.KV4_ERR_INVALID_ARG
    # off the default kernel the rotated query goes through `out` first, so an
    # `out` overlapping q is rejected before anything is launched
    lay2 = kv4.make_layout(max_seqs=2, num_pages=4, max_pages_per_seq=2)
    nws = kv4.workspace_bytes(lay2, 2)
    mem = ctypes.create_string_buffer(nws + 65536 + 16)
    b = (ctypes.addressof(mem) + 15) // 16 * 16
    ws = b + 65536
    prev = kv4.kv4_set_decode_kernel(kv4.KV4_KERNEL_MMA_SYNC)
    try:
        rc = lib.kv4_decode_attn_hadamard(ctypes.byref(lay2), b, b, b, b, 2, b, 0.1, 0, ws, nws,
                                          b + 64, None, None, None)
        assert rc == kv4.KV4_ERR_INVALID_ARG
    finally:
        kv4.kv4_set_decode_kernel(prev)


def test_fp4_entry_points_validate_on_host(lib):
    lay = kv4.make_layout(max_seqs=4, num_pages=10, max_pages_per_seq=4)
    # probe cache: 10 pages x 8 kv heads x (K, V) x 16 slots x (64 + 16) bytes
    assert kv4.fp4_cache_bytes(lay) == 10 * 8 * 2 * 16 * 80
    bad = kv4.make_layout(max_seqs=4, num_pages=10, max_pages_per_seq=4)
    bad.head_dim = 96
    assert kv4.fp4_cache_bytes(bad) == 0
    args = (None, None, None, None, None, 3, None, None, None, None)
    assert lib.kv4_fp4_append(ctypes.byref(lay), 3, 0, *args) == kv4.KV4_ERR_INVALID_ARG  # format
    assert lib.kv4_fp4_append(ctypes.byref(lay), 1, 0, *args) == kv4.KV4_ERR_INVALID_ARG  # NULLs
    assert lib.kv4_fp4_append(ctypes.byref(lay), 2, 1, None, None, None, None, None, 0, None,
                              None, None, None) == kv4.KV4_OK                             # T == 0
    assert lib.kv4_fp4_to_bf16(ctypes.byref(lay), 0, None, None, None) == kv4.KV4_ERR_INVALID_ARG
    assert lib.kv4_fp4_to_bf16(ctypes.byref(lay), 1, None, None, None) == kv4.KV4_ERR_INVALID_ARG


def test_diag_library_exports_its_header_and_validates_on_host():
    # the rate probe lives in its own library, declared in include/kv4_diag.h
    from int8_kv_cache_kv4_gb300 import build, diag
    if not os.path.exists(diag.LIB_PATH):
        build.build()
    dl = diag.load()
    names = diag.declared_symbols()
    assert names == ["kv4_diag_mma_rate"]
    for n in names:
        assert hasattr(dl, n)
    sink = ctypes.c_uint32(0)
    assert dl.kv4_diag_mma_rate(3, 1, 1, ctypes.addressof(sink), None) == 1  # no tcgen05 int8 kind
    assert dl.kv4_diag_mma_rate(0, 0, 1, ctypes.addressof(sink), None) == 1
    assert dl.kv4_diag_mma_rate(0, 1, 1, None, None) == 1
    assert not hasattr(lib_handle(), "kv4_diag_mma_rate")   # not in the decode library


def lib_handle():
    return kv4.load()
