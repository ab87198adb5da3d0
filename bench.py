#!/usr/bin/env python3
"""Benchmark of the GB300 FlashAttention-2 forward (one JSON line on stdout).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]
                  [--pass fwd|bwd]

A step is one forward pass (one kernel launch) over the workload's [B,H,N,D]
inputs, already resident in HBM. Timing uses CUDA events on the launching
stream around exactly K steps, bracketed by a barrier and a device
synchronise; the inputs rotate over enough copies that one pass over all of
them is larger than twice the L2 cache, so no step finds its inputs in L2
from the step before. The K steps are launched one by one through the
binding (--launch stream, the default); the same calls replayed from one
CUDA graph are timed after the timed region and reported beside it
("graph_replay"), which shows what the per-launch costs are worth on small
problems. Under torchrun the slowest rank's time is reported,
and the work is spread in one of two ways (--split):
  replicas  each rank runs the whole workload on its own GPU (weak scaling;
            the job's work grows with the number of ranks);
  heads     rank r of W owns a contiguous slice of the workload's B*H heads
            (attention_forward_03_gb300.partition.head_slice) and runs the
            forward on it alone (strong scaling: the job is one workload).
Neither puts a collective on the data path; --gather adds an all-gather of
the head slices' O and LSE to every step of the heads split.

Metric: attention forward TFLOP/s = 4*B*H*N^2*D (halved when causal) / time.
`--pass bwd` times the backward pass (fa2_bwd) instead: 10*B*H*N^2*D
(halved when causal) / time of the whole call.
`--impl reference` times the CPU fp64 oracle (this path's reference
implementation) on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "attention forward TFLOPS (4·B·H·N²·D) and % of GB300 dense fp16/bf16 peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = os.path.join(ROOT, "attention_forward_03_gb300", "csrc")


# ------------------------------------------------------------------ helpers
# the files that define the kernel and its device-resident launch (the
# host-memory pipeline and the no-allocation entry point do not change either)
KERNEL_FILES = ("fa2_kernel.cuh", "fa2_fwd_common.cuh", "fa2_launch.h", "sm103_ptx.cuh", "tmem_io.cuh",
                "fa2_fwd_d32.cu", "fa2_fwd_d64.cu", "fa2_fwd_d96.cu", "fa2_fwd_d128.cu", "fa2_api.cu")
# the head-dim-256 forward kernel
WIDE_KERNEL_FILES = ("fa2_kernel_wide.cuh", "fa2_fwd_common.cuh", "fa2_launch.h", "sm103_ptx.cuh", "tmem_io.cuh",
                     "fa2_fwd_d256.cu", "fa2_api.cu")
# the d-tiled forward kernel (head dims 512 and 1024)
DTILE_KERNEL_FILES = ("fa2_kernel_dtile.cuh", "fa2_fwd_common.cuh", "fa2_launch.h", "sm103_ptx.cuh", "tmem_io.cuh",
                      "fa2_fwd_d512.cu", "fa2_fwd_d1024.cu", "fa2_api.cu")
# the same for the backward pass (its three kernels and their launch)
BWD_KERNEL_FILES = ("fa2_bwd_kernel.cuh", "fa2_kernel.cuh", "fa2_fwd_common.cuh", "fa2_launch.h", "sm103_ptx.cuh",
                    "tmem_io.cuh", "fa2_bwd_d64.cu", "fa2_bwd_d128.cu", "fa2_bwd_api.cu", "fa2_api.cu")


def fwd_kernel_files(D: int):
    if D >= 512:
        return DTILE_KERNEL_FILES
    return WIDE_KERNEL_FILES if D == 256 else KERNEL_FILES


def kernel_source_hash(files=KERNEL_FILES) -> str:
    h = hashlib.sha256()
    for f in sorted(files):
        with open(os.path.join(KERNEL_SOURCES, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def traffic_per_launch(workload_name: str, files=KERNEL_FILES):
    """DRAM bytes per launch from a committed ncu capture, if it matches the current kernel source.
    Backward entries are keyed "bwd:<workload>"."""
    try:
        with open(PROFILE_TRAFFIC) as fh:
            t = json.load(fh)
    except (OSError, ValueError):
        return None
    entry = t.get(workload_name)
    if not entry or entry.get("kernel_source_hash") != kernel_source_hash(files):
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU is under load."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.t_start = None
        self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._reader = threading.Thread(target=self._read, daemon=True)
        self._reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t_start = time.time()

    def mark_stop(self):
        self.t_stop = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._reader.join(timeout=2)
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t_start and self.t_stop and self.t_start <= r[0] <= self.t_stop]
        used = inside if inside else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in used:
            for name, flag in zip(names, r[3][1:]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in used), "sm_max_mhz": max(r[2] for r in used),
                "reasons": sorted(reasons), "samples": len(used),
                "window": "timed region" if inside else "warm-up and timed region"}


# ------------------------------------------------------------- distributed
def dist_setup():
    """Return (rank, world, local_rank). Initialises torch.distributed under torchrun."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = os.environ.get("FA2_BENCH_BACKEND") or ("nccl" if torch.cuda.is_available() else "gloo")
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, world: int, max_seconds: float) -> float:
    """Weak scaling: every rank runs the whole workload; the job finishes with the slowest rank."""
    return flops_per_step * steps * world / max_seconds / 1e12


def split_job(w: workloads.Workload, split: str, world: int, rank: int):
    """This rank's share of the job: (local workload, first head, job FLOPs per step, parallelism label).

    replicas: the whole workload on every rank (the job does `world` of them).
    heads: flattened heads [h0, h1) of the one workload, run as a [1, h1 - h0, N, D]
    problem (the job does the workload once)."""
    import dataclasses

    from attention_forward_03_gb300 import partition
    if split == "replicas":
        return w, 0, workloads.flops(w) * world, f"weak x{world} (one independent replica per GPU)"
    h0, h1 = partition.head_slice(w.B * w.H, world, rank)
    local = dataclasses.replace(w, name=f"{w.name}[heads {h0}:{h1}]", B=1, H=h1 - h0)
    return local, h0, workloads.flops(w), f"heads x{world} (rank r owns a contiguous slice of the B*H heads)"


def time_steps(step, steps: int, stream, dev, launch: str, clocks=None, resettle_s: float = 0.5) -> float:
    """Device seconds for `steps` calls of step(i, stream), on `stream`, by CUDA events.

    launch="stream": the calls are made one by one inside the timed region.
    launch="graph": the same calls (through the same API, with the same
    arguments) are captured once into a CUDA graph on a side stream and the
    graph is replayed once inside the timed region, so the per-launch host and
    launch-queue costs are not in the timing; every step's kernels still run.
    """
    import torch
    if launch == "graph":
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            step(0, cap)  # per-stream set-up (the binding's cached workspace) before the capture
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for i in range(steps):
                step(i, cap)
        # untimed replays: the first pays the graph's upload, and the clocks,
        # which drop while the GPU idles during the capture, ramp back up
        # (a timed replay straight after the capture measured 5-8 % low)
        t0 = time.perf_counter()
        while True:
            with torch.cuda.stream(stream):
                g.replay()
            torch.cuda.synchronize(dev)
            if time.perf_counter() - t0 >= resettle_s:
                break
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    if clocks is not None:
        clocks.mark_start()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        if launch == "graph":
            g.replay()
        else:
            for i in range(steps):
                step(i, stream)
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    if clocks is not None:
        clocks.mark_stop()
    return ev0.elapsed_time(ev1) / 1e3


# ------------------------------------------------------------- CPU oracle leg
def _row_flops(w: workloads.Workload, rows):
    import numpy as np
    rows = np.asarray(rows)
    if not w.causal:
        return 4.0 * w.D * w.N * len(rows)
    return float(np.sum(4.0 * w.D * np.minimum(w.N, rows % w.N + 1)))


def oracle_rows(w: workloads.Workload, target_seconds: float, inputs):
    """Rows of a bounded oracle sample of the workload: a uniform random subset
    of all B*H*N query rows sized so that one oracle call on it takes about
    `target_seconds` (None = the whole workload, when that fits). The rate is
    calibrated on growing probes until one runs for about a second, so that
    per-call fixed costs do not dominate it."""
    import numpy as np

    import oracle
    q, k, v = inputs
    threads = oracle.default_threads()
    total = w.B * w.H * w.N
    per_row = workloads.flops(w) / total
    rng = np.random.default_rng(0)
    size = min(total, 2 * threads)
    while True:
        probe = np.sort(rng.choice(total, size=size, replace=False))
        t0 = time.perf_counter()
        oracle.attention_fwd(q, k, v, w.scale, w.causal, rows=probe, nthreads=threads)
        took = max(time.perf_counter() - t0, 1e-4)
        rate = _row_flops(w, probe) / took
        if took >= min(1.0, target_seconds / 4) or size >= total:
            break
        size = int(min(total, max(2 * size, size * min(1.0, target_seconds / 4) / took)))
    want = int(min(total, max(threads, target_seconds * rate / per_row)))
    return np.sort(rng.choice(total, size=want, replace=False)) if want < total else None


def host_cpu_model() -> str:
    """The host CPU's model (best effort from /proc/cpuinfo: the model name where
    there is one, else the Arm implementer and part codes)."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                key, _, val = line.partition(":")
                key, val = key.strip().lower(), val.strip()
                if val and key not in fields:
                    fields[key] = val
    except OSError:
        pass
    for key in ("model name", "cpu model", "hardware"):
        if key in fields:
            return fields[key]
    if "cpu part" in fields:
        return f"{platform.machine()} (CPU implementer {fields.get('cpu implementer', '?')}, part {fields['cpu part']})"
    return platform.processor() or platform.machine()


def time_oracle(w: workloads.Workload, rows, inputs):
    """One timed oracle call on `rows` (None = every row).
    Returns (tflops, seconds, rows, threads, description)."""
    import oracle
    q, k, v = inputs
    threads = oracle.default_threads()
    total = w.B * w.H * w.N
    t0 = time.perf_counter()
    oracle.attention_fwd(q, k, v, w.scale, w.causal, rows=rows, nthreads=threads)
    secs = time.perf_counter() - t0
    n = total if rows is None else len(rows)
    fl = workloads.flops(w) if rows is None else _row_flops(w, rows)
    what = "the whole workload" if rows is None else f"{n} of its {total} query rows, drawn uniformly"
    desc = f"{what} ({w.describe()}, each row over its full allowed key range), fp64, {threads} threads"
    return fl / secs / 1e12, secs, n, threads, desc


def oracle_sample(w: workloads.Workload, target_seconds: float, inputs=None):
    """Time the fp64 oracle on a bounded sample of about `target_seconds`."""
    inputs = inputs if inputs is not None else workloads.make_inputs(w)
    return time_oracle(w, oracle_rows(w, target_seconds, inputs), inputs)


# -------------------------------------------------------------------- arms
def run_reference(args, w, rank, world):
    if rank != 0:
        return None
    import numpy as np  # noqa: F401
    # one sample of rows, sized once, timed every step: the whole run takes
    # about reference_seconds plus the calibration
    per_step = max(0.05, args.reference_seconds / max(1, args.steps + args.warmup))
    inputs = workloads.make_inputs(w)
    rows = oracle_rows(w, per_step, inputs)
    for _ in range(args.warmup):
        time_oracle(w, rows, inputs)
    vals, secs = [], []
    desc, threads = "", 1
    for _ in range(args.steps):
        tf, s, n, threads, desc = time_oracle(w, rows, inputs)
        vals.append(tf)
        secs.append(s)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0, sigma^2) inputs, cast to the workload's 16-bit dtype)",
        "config": {"workload": w.describe(), "B": w.B, "H": w.H, "N": w.N, "D": w.D, "causal": w.causal,
                   "input_dtype": w.dtype, "l2": "host CPU run; no GPU L2 involved"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "cpu_model": host_cpu_model(), "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def run_gb300(args, w, rank, world, local):
    import torch

    import attention_forward_03_gb300 as fa2
    if not torch.cuda.is_available():
        raise RuntimeError("the gb300 arm needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa2.library()
    stream = torch.cuda.current_stream(dev)

    from attention_forward_03_gb300 import partition
    job = w
    w, h0, job_flops, parallelism = split_job(job, args.split, world, rank)
    q, k, v = workloads.make_inputs(job)
    if args.split == "heads":
        q, k, v = (partition.local_view(t, h0, h0 + w.H).contiguous() for t in (q, k, v))
    resolved_schedule = args.schedule
    if resolved_schedule == "auto":
        resolved_schedule = fa2.binding.choose_schedule(w.B, w.H, w.N, w.causal,
                                                        torch.cuda.get_device_properties(dev).multi_processor_count,
                                                        w.D)
    set_bytes = max(1, workloads.algorithmic_bytes(w))
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 * 2 ** 20)
    nsets = max(2, math.ceil(2 * l2 / set_bytes))
    sets = []
    for _ in range(nsets):
        sets.append((q.to(dev), k.to(dev), v.to(dev), torch.empty_like(q, device=dev),
                     torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)))
    torch.cuda.synchronize(dev)

    gather = args.gather and args.split == "heads" and world > 1

    launch = "stream" if gather else args.launch

    def step(i, st=None):
        qd, kd, vd, od, ld = sets[i % nsets]
        fa2.attention_forward(qd, kd, vd, scale=w.scale, is_causal=w.causal, out=od, lse=ld,
                              stream=st if st is not None else stream, schedule=args.schedule)
        if gather:
            partition.gather_heads(od, job.B * job.H, world, rank)
            partition.gather_heads(ld, job.B * job.H, world, rank)

    clocks = ClockSampler(local)
    clocks.start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    # keep the GPU busy for ~1 s before the timed region so clocks settle and get sampled
    t0 = time.perf_counter()
    i = 0
    while time.perf_counter() - t0 < args.settle_seconds:
        step(i)
        i += 1
        if i % 16 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    fa2.fa2_device_status(clear=True)

    barrier(world)
    elapsed = time_steps(step, args.steps, stream, dev, launch, clocks)
    barrier(world)
    clock_info = clocks.stop()
    status = fa2.fa2_device_status(clear=True)
    if status != 0:
        raise RuntimeError(f"device watchdog fired during the timed region (code {status})")
    # the same steps the other way (reported beside the headline, not in it)
    other = "graph" if launch == "stream" else "stream"
    other_elapsed = None if gather else time_steps(step, args.steps, stream, dev, other)
    t_max = max_over_ranks(elapsed, world, dev)
    t_max_other = None if other_elapsed is None else max_over_ranks(other_elapsed, world, dev)
    flops = workloads.flops(w)  # this rank's launches
    value = job_flops * args.steps / t_max / 1e12
    per_launch = elapsed / args.steps

    # End to end through the C ABI's host-memory entry point (fa2_fwd_host):
    # page-locked host buffers in, host buffers out, every copy inside the
    # timed region, chunks of heads pipelined over the copy engines.
    # Q, K, V in one page-locked [3, B, H, N, D] buffer (a fused QKV
    # projection's layout): the call then moves each chunk's three blocks in
    # one 2-D copy; LSE in page-locked memory is written by the kernels.
    qkv_h = torch.empty((3, *q.shape), dtype=q.dtype).pin_memory()
    for i, t in enumerate((q, k, v)):
        qkv_h[i].copy_(t)
    qh, kh, vh = qkv_h[0], qkv_h[1], qkv_h[2]
    oh = torch.empty_like(q).pin_memory()
    lh = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
    del sets
    torch.cuda.empty_cache()
    host_buf = torch.empty(fa2.fa2_fwd_host_buffer_bytes(w.B, w.H, w.N, w.D), dtype=torch.uint8, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    hpc = args.e2e_heads_per_chunk or fa2.binding.host_chunk_heads(w.B, w.H, w.N, w.causal, sms, w.D)
    chunk_schedule = args.schedule
    if chunk_schedule == "auto":
        chunk_schedule = fa2.binding.choose_schedule(1, min(hpc, w.B * w.H), w.N, w.causal, sms, w.D)

    def e2e_step():
        fa2.attention_forward_host(qh, kh, vh, scale=w.scale, is_causal=w.causal, out=oh, lse=lh, stream=stream,
                                   device=dev, heads_per_chunk=hpc, schedule=chunk_schedule,
                                   device_buffer=host_buf, synchronize=False)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_steps = max(3, min(args.steps, 50))
    barrier(world)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_elapsed = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, world, dev)
    e2e_value = job_flops * e2e_steps / e2e_elapsed / 1e12
    # bytes of the whole job (all ranks)
    copies = world if args.split == "replicas" else 1
    jq = job.B * job.H * job.N * job.D * q.element_size()
    h2d = 3 * jq * copies
    d2h = (jq + job.B * job.H * job.N * 4) * copies

    if rank != 0:
        return None
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops / per_launch / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps, "higher_is_better": True,
        "scaling": "weak" if args.split == "replicas" else "strong", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded N(0, sigma^2) inputs, cast to the workload's 16-bit dtype)",
        "config": {"workload": job.describe(), "B": job.B, "H": job.H, "N": job.N, "D": job.D,
                   "causal": job.causal, "scale": "1/sqrt(D)", "schedule": resolved_schedule,
                   "parallelism": parallelism + (", O/LSE all-gathered every step" if gather else ""),
                   "rank0_heads": [h0, h0 + w.B * w.H] if args.split == "heads" else None,
                   "launch": ("one CUDA graph of the K steps' launches (captured through the binding and the "
                              "C ABI), replayed once" if launch == "graph" else "K launches made one by one"),
                   "l2": f"inputs rotate over {nsets} copies ({nsets * set_bytes / 2**20:.0f} MiB > 2x L2)"},
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": f"{peak_src} bf16 dense (burst)",
                     "traffic": traffic_per_launch(w.name, fwd_kernel_files(w.D)),
                     "algorithmic_bytes": workloads.algorithmic_bytes(w),
                     "achieved_hbm_gbs": workloads.algorithmic_bytes(w) / per_launch / 1e9},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "fa2_fwd_host (C ABI, page-locked host buffers)",
                "host_layout": "Q, K, V packed in one [3, B, H, N, D] buffer; LSE written in place by the kernels",
                "heads_per_chunk": hpc,
                "chunk_schedule": chunk_schedule, "steps": e2e_steps},
        "gpu_launches": args.steps if w.B * w.H > 0 else 0,
        "clocks": clock_info,
        ("graph_replay" if other == "graph" else "stream_launch"): None if t_max_other is None else {
            "value": job_flops * args.steps / t_max_other / 1e12, "unit": UNIT,
            "ms_per_step": 1e3 * t_max_other / args.steps,
            "what": ("the same K steps' calls captured into one CUDA graph and replayed (no per-launch host or "
                     "queue cost), measured after the timed region" if other == "graph" else
                     "the same K steps launched one by one from the host, measured after the timed region")},
    }
    if not args.no_cpu_baseline:
        tf, secs, rows, threads, desc = oracle_sample(job, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tf, "unit": UNIT, "cores": threads, "cpu_model": host_cpu_model(), "kind": "oracle", "sample": desc,
                                "seconds": secs}
    return line


BWD_METRIC = "attention backward TFLOPS (10·B·H·N²·D: S, dP, dV, dK, dQ products) and % of GB300 dense fp16/bf16 peak"


def time_grad_oracle(w: workloads.Workload, heads, inputs):
    """One timed gradient-oracle call on whole heads. Returns (tflops, seconds, threads, description)."""
    import oracle
    q, k, v, do = inputs
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.attention_bwd(q, k, v, do, w.scale, w.causal, heads=heads, nthreads=threads)
    secs = time.perf_counter() - t0
    fl = workloads.bwd_flops(w) * len(heads) / (w.B * w.H)
    desc = (f"{len(heads)} of its {w.B * w.H} heads, whole ({w.describe()}), gradient of the fp64 definition, "
            f"{threads} threads")
    return fl / secs / 1e12, secs, threads, desc


def run_gb300_bwd(args, w, rank, world, local):
    """The backward pass (fa2_bwd: row-statistics prologue, backward kernel, dQ conversion) as the step."""
    import torch

    import attention_forward_03_gb300 as fa2
    if not torch.cuda.is_available():
        raise RuntimeError("the gb300 arm needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa2.library()
    stream = torch.cuda.current_stream(dev)
    q, k, v = workloads.make_inputs(w)
    do = workloads.make_grad_output(w)
    set_bytes = workloads.bwd_algorithmic_bytes(w)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 * 2 ** 20)
    nsets = max(2, math.ceil(2 * l2 / set_bytes))
    need = fa2.fa2_bwd_workspace_bytes(w.B, w.H, w.N, w.D)
    sets = []
    for _ in range(nsets):
        qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
        od, ld = fa2.attention_forward(qd, kd, vd, scale=w.scale, is_causal=w.causal, stream=stream)
        outs = tuple(torch.empty_like(qd) for _ in range(3))
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        sets.append((qd, kd, vd, od, ld, dod, outs, ws))
    torch.cuda.synchronize(dev)

    def step(i, st=None):
        qd, kd, vd, od, ld, dod, outs, ws = sets[i % nsets]
        fa2.attention_backward(qd, kd, vd, od, ld, dod, scale=w.scale, is_causal=w.causal, dq=outs[0], dk=outs[1],
                               dv=outs[2], workspace=ws, stream=st if st is not None else stream,
                               schedule=args.schedule)

    clocks = ClockSampler(local)
    clocks.start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    i = 0
    while time.perf_counter() - t0 < args.settle_seconds:
        step(i)
        i += 1
        if i % 8 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    fa2.fa2_device_status(clear=True)
    barrier(world)
    elapsed = time_steps(step, args.steps, stream, dev, args.launch, clocks)
    barrier(world)
    clock_info = clocks.stop()
    status = fa2.fa2_device_status(clear=True)
    if status != 0:
        raise RuntimeError(f"device watchdog fired during the timed region (code {status})")
    t_max = max_over_ranks(elapsed, world, dev)
    flops = workloads.bwd_flops(w)
    value = whole_job_tflops(flops, args.steps, world, t_max)
    per_call = elapsed / args.steps
    if rank != 0:
        return None
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops / per_call / 1e12
    line = {
        "pass": "backward", "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded N(0, sigma^2) Q, K, V and dO, cast to the workload's 16-bit dtype; "
                "O and LSE from fa2_fwd)",
        "config": {"workload": w.describe(), "B": w.B, "H": w.H, "N": w.N, "D": w.D, "causal": w.causal,
                   "scale": "1/sqrt(D)", "schedule": args.schedule + (" (the library's choice)"
                                                                      if args.schedule == "auto" else ""),
                   "parallelism": f"weak x{world} (one independent replica per GPU)",
                   "launch": ("one CUDA graph of the K steps' calls, replayed once" if args.launch == "graph"
                              else "K calls made one by one"),
                   "l2": f"inputs rotate over {nsets} copies ({nsets * set_bytes / 2**20:.0f} MiB > 2x L2)"},
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": f"{peak_src} bf16 dense (burst)",
                     "timed": "the whole fa2_bwd call (prologue, backward kernel and dQ conversion)",
                     "traffic": traffic_per_launch("bwd:" + w.name, BWD_KERNEL_FILES),
                     "traffic_of": "fa2_bwd_kernel (97.5% of the call's device time)",
                     "algorithmic_bytes": set_bytes,
                     "achieved_hbm_gbs": set_bytes / per_call / 1e9},
        "gpu_launches": 3 * args.steps,
        "clocks": clock_info,
    }
    if not args.no_cpu_baseline:
        tf, secs, threads, desc = time_grad_oracle(w, [0], (q, k, v, do))
        line["cpu_baseline"] = {"value": tf, "unit": UNIT, "cores": threads, "cpu_model": host_cpu_model(), "kind": "oracle", "sample": desc,
                                "seconds": secs}
    return line


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="target", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--schedule", default="auto", choices=["auto", "balanced", "units"],
                    help="forward: auto = the binding's choice, balanced = fa2_fwd_ws (equal K/V-tile steps per "
                         "SM), units = fa2_fwd; backward (--pass bwd): the same choice passed to fa2_bwd_sched "
                         "(auto = the library's)")
    ap.add_argument("--split", default="replicas", choices=["replicas", "heads"],
                    help="under torchrun: replicas = every rank runs the whole workload (weak scaling); heads = "
                         "rank r owns a contiguous slice of the B*H heads (strong scaling)")
    ap.add_argument("--gather", action="store_true",
                    help="with --split heads: all-gather O and LSE of every step to every rank (NCCL)")
    ap.add_argument("--launch", default="stream", choices=["stream", "graph"],
                    help="stream: the K timed steps are launched one by one through the binding; graph: the same "
                         "calls captured once into a CUDA graph and replayed (no per-launch host or queue cost). "
                         "The other one is measured after the timed region and reported beside it")
    ap.add_argument("--settle-seconds", type=float, default=1.0)
    ap.add_argument("--e2e-heads-per-chunk", type=int, default=0,
                    help="heads per chunk of the end-to-end host-memory pipeline (0 = the binding's default)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reference-seconds", type=float, default=120.0,
                    help="total CPU time budget of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="which", default="fwd", choices=["fwd", "bwd"],
                    help="fwd: the forward pass (the headline); bwd: the backward pass (fa2_bwd)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = workloads.WORKLOADS[args.workload]
    if args.impl == "reference" and args.which == "bwd":
        ap.error("--impl reference times the forward oracle; the backward's CPU baseline is in its gb300 line")
    if args.impl == "reference":
        # the CPU oracle runs on rank 0 only; other ranks exit without work
        rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
        line = run_reference(args, w, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    rank, world, local = dist_setup()
    if world != args.gpus and rank == 0:
        print(f"note: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    line = (run_gb300_bwd if args.which == "bwd" else run_gb300)(args, w, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
