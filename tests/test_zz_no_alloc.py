"""The decode entry point for callers that cannot allocate device memory.

Such callers (a plug-in whose host framework has reserved all free device
memory, a decode loop that must not call cudaMalloc because it synchronises
the device, a runtime without a device allocator) use
kv4_decode_attn_noalloc, which takes its workspace from a fixed scratch array
inside the library.  Its output must match kv4_decode_attn's on the same
inputs, call after call (the shared scratch keeps the previous call's
contents, so a second call checks that nothing stale leaks in).  Both entry
points run the same deterministic kernels, so the outputs must agree bit for
bit.  This file is collected last so that a failure here leaves every other
test already run.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from kv4_case import Case  # noqa: E402
from int8_kv_cache_kv4_gb300 import kv4  # noqa: E402


def _decode(c, gc, noalloc, max_splits=0):
    """One decode of case c; the workspace path gets a fresh workspace."""
    dev = gc.device
    q = torch.from_numpy(c.q.view(np.int16)).to(dev).view(torch.bfloat16)
    lens = torch.from_numpy(c.lens).to(dev)
    out = torch.full((c.B, c.h_q, c.d_h), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((c.B, c.h_q), float("nan"), dtype=torch.float32, device=dev)
    if noalloc:
        kv4.kv4_decode_attn_noalloc(gc.layout, gc.paged, gc.side, q, lens, gc.block_table, out,
                                    lse, gc.sm_scale, max_splits, gc.status)
    else:
        ws = torch.full((kv4.workspace_bytes(gc.layout, c.B, max_splits),), 0x5A, dtype=torch.uint8,
                        device=dev)
        kv4.kv4_decode_attn(gc.layout, gc.paged, gc.side, q, lens, gc.block_table, ws, out, lse,
                            gc.sm_scale, max_splits, gc.status)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy(), lse.cpu().numpy()


def test_noalloc_decode_matches_workspace_decode_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kv4.load(build_if_missing=True)
    c = Case([300, 1000, 77, 2000, 1, 513], S=4, R=64, g=32, seed=21)
    gc = c.gpu()
    ref_o, ref_l = _decode(c, gc, noalloc=False)
    for _ in range(2):
        o, l = _decode(c, gc, noalloc=True)
        assert np.array_equal(o, ref_o), "outputs differ from kv4_decode_attn's"
        assert np.array_equal(l, ref_l), "log-normalisers differ from kv4_decode_attn's"
    assert gc.read_status() == 0


def test_noalloc_after_a_larger_call_and_on_every_kernel():
    # The completion counters sit after the partial outputs, at an offset that
    # moves with the call's size: a large call, then smaller ones -- the
    # default kernel, the split kernel (max_splits > 0, counters cleared by the
    # entry point) and the CUDA-core kernel -- must each match a fresh-workspace
    # call bit for bit.
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kv4.load(build_if_missing=True)
    big = Case([900] * 40 + [3000, 17, 1], S=4, R=64, g=32, seed=31)
    small = Case([700, 33, 2100], S=4, R=64, g=32, seed=32)
    gb, gs = big.gpu(), small.gpu()
    o, _ = _decode(big, gb, noalloc=True)
    assert np.array_equal(o, _decode(big, gb, noalloc=False)[0])
    prev = kv4.kv4_set_decode_kernel(kv4.KV4_KERNEL_AUTO)
    try:
        for which, ms in ((kv4.KV4_KERNEL_AUTO, 0), (kv4.KV4_KERNEL_AUTO, 3),
                          (kv4.KV4_KERNEL_CUDA_CORE, 0)):
            kv4.kv4_set_decode_kernel(which)
            ref_o, ref_l = _decode(small, gs, noalloc=False, max_splits=ms)
            for _ in range(2):
                o, l = _decode(small, gs, noalloc=True, max_splits=ms)
                assert np.array_equal(o, ref_o), f"kernel {which}, max_splits {ms}"
                assert np.array_equal(l, ref_l), f"kernel {which}, max_splits {ms}"
            _decode(big, gb, noalloc=True)   # leave the large call's contents behind
    finally:
        kv4.kv4_set_decode_kernel(prev)
    assert gb.read_status() == 0 and gs.read_status() == 0


def test_noalloc_rejects_requests_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kv4.load(build_if_missing=True)
    cap = kv4.load().kv4_noalloc_scratch_bytes()
    # a batch whose partial outputs alone exceed the scratch
    lay = kv4.make_layout(sink=0, recent=0, max_seqs=4096, num_pages=64, max_pages_per_seq=4096)
    assert kv4.workspace_bytes(lay, 4096) > cap
    dev = torch.device("cuda")
    q = torch.zeros((4096, 32, 128), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    lens = torch.zeros(4096, dtype=torch.int32, device=dev)
    bt = torch.zeros((4096, 4096), dtype=torch.int32, device=dev)
    paged = torch.zeros(kv4.paged_cache_bytes(lay), dtype=torch.uint8, device=dev)
    side = torch.zeros(16, dtype=torch.uint8, device=dev)
    with pytest.raises(kv4.KV4Error, match="workspace"):
        kv4.kv4_decode_attn_noalloc(lay, paged, side, q, lens, bt, out)


def test_decode_bindings_reject_missized_tensors():
    # a tensor that does not match the layout and q is refused on the host
    # (KV4Error), before anything reaches the device
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kv4.load(build_if_missing=True)
    c = Case([40, 9], S=4, R=16, g=32, seed=33)
    gc = c.gpu()
    dev = gc.device
    q = torch.zeros((c.B, c.h_q, c.d_h), dtype=torch.bfloat16, device=dev)
    lens = torch.from_numpy(c.lens).to(dev)
    good = dict(out=torch.empty_like(q), out_lse=torch.empty((c.B, c.h_q), device=dev))
    bad_cases = [
        dict(good, out=torch.empty((c.B, c.h_q, c.d_h - 1), dtype=torch.bfloat16, device=dev)),
        dict(good, out_lse=torch.empty((c.B + 1, c.h_q), device=dev)),
    ]
    for kw in bad_cases:
        with pytest.raises(kv4.KV4Error):
            kv4.kv4_decode_attn_noalloc(gc.layout, gc.paged, gc.side, q, lens, gc.block_table, **kw)
    with pytest.raises(kv4.KV4Error):   # seq_lens shorter than the batch
        kv4.kv4_decode_attn_noalloc(gc.layout, gc.paged, gc.side, q, lens[:1], gc.block_table, **good)
    with pytest.raises(kv4.KV4Error):   # block table not [max_seqs][max_pages_per_seq]
        kv4.kv4_decode_attn_noalloc(gc.layout, gc.paged, gc.side, q, lens, gc.block_table[:, :1],
                                    **good)
    ws = torch.empty(kv4.workspace_bytes(gc.layout, c.B), dtype=torch.uint8, device=dev)
    with pytest.raises(kv4.KV4Error):
        kv4.kv4_decode_attn(gc.layout, gc.paged, gc.side, q[:, :8], lens, gc.block_table, ws,
                            good["out"])
