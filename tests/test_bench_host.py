"""Host-side arithmetic of the benchmark (no GPU): the algorithmic bytes the
roofline divides by, counted two independent ways, and the workload sizes
the bench line names."""
import numpy as np

import bench
from int8_kv_cache_kv4_gb300 import rollout as R
from int8_kv_cache_kv4_gb300 import workloads as W


def test_decode_bytes_agree_between_bench_and_driver():
    for name in ("tiny_b4_l512", "qwen3_8b_b64", "long_128k"):
        w = W.WORKLOADS[name]
        lens = W.seq_lengths(w)
        dec, _, n4, n8 = bench.algorithmic_bytes(lens, w)
        per = R.decode_bytes(lens[None, :], h_q=w.h_q, h_kv=w.h_kv, d_h=w.d_h, group=w.group,
                             sink=w.sink, recent=w.recent)
        assert int(per[0]) == dec, name
        assert n4 + n8 == int(lens.sum())


def test_batch64_layer_bytes():
    # 64 sequences, U[1024, 8192]: 386.3 MB per decode, about 95 % of it INT4
    w = W.WORKLOADS["qwen3_8b_b64"]
    lens = W.seq_lengths(w)
    dec, app, n4, n8 = bench.algorithmic_bytes(lens, w)
    assert dec == 386305328
    assert n8 == 64 * (w.sink + w.recent)
    assert 0.94 < n4 * 8 * 160 / dec < 0.96
    # append: bf16 K/V read, INT4 and INT8 entries written, three int32 per token
    assert app == 64 * 8 * (512 + 160 + 260) + 64 * 12


def test_kernel_source_hash_is_stable():
    h = bench.kernel_source_hash()
    assert len(h) == 16 and h == bench.kernel_source_hash()
    assert all(isinstance(k, tuple) and len(k) == 2 for k in bench.TRAFFIC)
