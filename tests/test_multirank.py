"""World-size-2 checks (gloo, CPU) of the benchmark's multi-rank host logic: the
barrier, the max-over-ranks timing and the whole-job (weak-scaling) aggregate."""
from __future__ import annotations

import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "FA2_BENCH_BACKEND": "gloo"})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    elapsed = 1.0 + rank  # rank 1 is the slower one
    t_max = bench.max_over_ranks(elapsed, w)
    value = bench.whole_job_tflops(2e12, 10, w, t_max)
    q.put((rank, t_max, value))
    dist.destroy_process_group()


def test_two_ranks_report_the_slowest_rank_and_the_whole_job():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, t_max, value in got:
        assert t_max == 2.0
        # 2 ranks x 10 steps x 2 TFLOP in 2 s = 20 TFLOP/s
        assert abs(value - 20.0) < 1e-9


def test_single_rank_needs_no_process_group(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup() == (0, 1, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_tflops(1e12, 4, 1, 2.0) == 2.0
