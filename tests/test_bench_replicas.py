"""The N > 1 path of bench.py on CPU: world_size-2 gloo ranks, each with its
own timing, must all see the slowest rank's time, and the whole-job value must
count every replica's tokens.  The reference arm prints only on rank 0."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [3.0, 5.0][rank]
    got = bench.reduce_max_ms(local_ms, world, torch.device("cpu"))
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got, bench.replica_value(world, 1000, got / 10)))


def test_two_rank_max_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [5.0, 5.0]          # both ranks see the slowest
    assert all(abs(r[2] - 2 * 1000 / 0.5e-3) < 1e-6 for r in res)  # 2 replicas x 1000 tokens / 0.5 ms


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"workload": "tiny_b4_l512", "steps": 1, "warmup": 0, "cpu_budget": 0.1})()
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    assert buf.getvalue() == ""
