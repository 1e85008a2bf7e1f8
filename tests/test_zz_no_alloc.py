"""The decode entry point for callers that cannot allocate device memory.

Such callers (a plug-in whose host framework has reserved all free device
memory, a decode loop that must not call cudaMalloc because it synchronises
the device, a runtime without a device allocator) use
kv4_decode_attn_noalloc, which takes its workspace from a fixed scratch array
inside the library.  Its output must match kv4_decode_attn's on the same
inputs, call after call (the shared scratch keeps the previous call's
contents, so a second call checks that nothing stale leaks in).  This file is
collected last so that a failure here leaves every other test already run.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from kv4_case import Case, MAX_ABS  # noqa: E402
from int8_kv_cache_kv4_gb300 import kv4  # noqa: E402


def _decode(c, gc, noalloc):
    dev = gc.device
    q = torch.from_numpy(c.q.view(np.int16)).to(dev).view(torch.bfloat16)
    lens = torch.from_numpy(c.lens).to(dev)
    out = torch.full((c.B, c.h_q, c.d_h), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((c.B, c.h_q), float("nan"), dtype=torch.float32, device=dev)
    if noalloc:
        kv4.kv4_decode_attn_noalloc(gc.layout, gc.paged, gc.side, q, lens, gc.block_table, out,
                                    lse, gc.sm_scale, 0, gc.status)
    else:
        gc.decode(q, lens, out, lse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def test_noalloc_decode_matches_workspace_decode_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kv4.load(build_if_missing=True)
    c = Case([300, 1000, 77, 2000, 1, 513], S=4, R=64, g=32, seed=21)
    gc = c.gpu()
    ref_o, ref_l = _decode(c, gc, noalloc=False)
    for _ in range(2):
        o, l = _decode(c, gc, noalloc=True)
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
        assert np.max(np.abs(o - ref_o)) <= MAX_ABS
        assert np.max(np.abs(l - ref_l)) <= 1e-3
    assert gc.read_status() == 0


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
