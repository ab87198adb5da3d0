"""The multi-GPU partition of the forward pass by heads (host logic), checked on
CPU: slices of the flattened B*H heads, their byte offsets, and the optional
all-gather of the sharded outputs with gloo ranks (world sizes 2 and 3)."""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from attention_forward_03_gb300 import partition  # noqa: E402


@pytest.mark.parametrize("total", [0, 1, 2, 3, 7, 8, 64, 97, 192])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_every_head_owned_once_contiguous_and_balanced(total, world):
    slices = [partition.head_slice(total, world, r) for r in range(world)]
    assert slices[0][0] == 0 and slices[-1][1] == total
    for (a0, a1), (b0, b1) in zip(slices, slices[1:]):
        assert a1 == b0  # contiguous, in rank order, no overlap and no gap
    sizes = [b - a for a, b in slices]
    assert all(s >= 0 for s in sizes) and sum(sizes) == total
    assert max(sizes) - min(sizes) <= 1  # balanced
    assert sizes == sorted(sizes, reverse=True)  # the extra heads go to the first ranks
    owners = [r for r, (a, b) in enumerate(slices) for _ in range(a, b)]
    assert owners == sorted(owners) and len(owners) == total


def test_bad_slice_arguments():
    for args in ((-1, 2, 0), (4, 0, 0), (4, 2, 2), (4, 2, -1)):
        with pytest.raises(ValueError):
            partition.head_slice(*args)


def test_slice_bytes_address_the_right_rows():
    B, H, N, D = 2, 3, 5, 8
    t = torch.arange(B * H * N * D, dtype=torch.int16).reshape(B, H, N, D)
    raw = t.numpy().tobytes()
    for world in (2, 3, 4):
        for r in range(world):
            a, b = partition.head_slice(B * H, world, r)
            off = partition.slice_bytes(a, b, N, D)
            view = partition.local_view(t, a, b)
            assert view.shape == (1, b - a, N, D)
            assert raw[off["tensor_offset"]:off["tensor_offset"] + off["tensor_bytes"]] == \
                view.contiguous().numpy().tobytes()
            lse = torch.arange(B * H * N, dtype=torch.float32).reshape(B, H, N)
            lraw = lse.numpy().tobytes()
            lv = partition.local_view(lse, a, b)
            assert lraw[off["lse_offset"]:off["lse_offset"] + off["lse_bytes"]] == lv.contiguous().numpy().tobytes()


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "FA2_BENCH_BACKEND": "gloo"})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    import workloads
    from attention_forward_03_gb300 import partition as part
    r, w, _ = bench.dist_setup()
    out = {}
    # uneven split: 7 heads of N=5, D=4 over w ranks; each rank "computes" its
    # slice (here: a function of the global head index) and the gather
    # reassembles the full tensor in head order on every rank
    B, H, N, D = 1, 7, 5, 4
    a, b = part.head_slice(B * H, w, r)
    glob = torch.arange(B * H * N * D, dtype=torch.float32).reshape(B, H, N, D) * 0.5
    local = part.local_view(glob, a, b).contiguous()
    full = part.gather_heads(local, B * H, w, r)
    out["gather_ok"] = bool(torch.equal(full, glob.reshape(B * H, N, D)))
    lse = torch.arange(B * H * N, dtype=torch.float32).reshape(B, H, N) - 3.0
    full_lse = part.gather_heads(part.local_view(lse, a, b).contiguous(), B * H, w, r)
    out["gather_lse_ok"] = bool(torch.equal(full_lse, lse.reshape(B * H, N)))
    # the benchmark's share of the job: heads split = one workload in all
    job = workloads.WORKLOADS["ragged"]
    local_w, h0, job_flops, label = bench.split_job(job, "heads", w, r)
    out["share"] = (h0, local_w.B, local_w.H, local_w.N, local_w.D)
    out["job_flops"] = job_flops
    rep_w, _, rep_flops, _ = bench.split_job(job, "replicas", w, r)
    out["replica"] = (rep_w == job, rep_flops == workloads.flops(job) * w)
    # max over ranks of the elapsed time, and the whole job's rate from it
    t_max = bench.max_over_ranks(1.0 + r, w)
    out["t_max"] = t_max
    q.put((r, out))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_split_the_heads_and_gather_them(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    got = dict(q.get(timeout=5) for _ in range(world))
    import workloads
    job = workloads.WORKLOADS["ragged"]
    heads = 0
    for r in range(world):
        o = got[r]
        assert o["gather_ok"] and o["gather_lse_ok"]
        h0, B, H, N, D = o["share"]
        assert (h0, h0 + H) == partition.head_slice(job.B * job.H, world, r)
        assert B == 1 and N == job.N and D == job.D
        heads += H
        assert o["job_flops"] == workloads.flops(job)  # the job is the workload once, not per rank
        assert o["replica"] == (True, True)
        assert o["t_max"] == float(world)
    assert heads == job.B * job.H
