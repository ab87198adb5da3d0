"""Parity of the sm_103a forward kernel with the CPU fp64 oracle, through the C ABI.

Tolerances (max-abs, GPU output vs the fp64 oracle on the same seeded 16-bit
inputs): O within 2e-3 for fp16 and 1e-2 for bf16, LSE within 1e-3.
Small shapes are compared element by element on every row; the full-size
workloads, launched exactly as the benchmark launches them, are compared on
a sample of rows (random rows plus the first/last rows of heads and rows on
both sides of tile boundaries).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

TOL_O = {"f16": 2e-3, "bf16": 1e-2}
TOL_LSE = 1e-3


@pytest.fixture(scope="module")
def fa2():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from attention_forward_03_gb300 import build
    build.build()
    import attention_forward_03_gb300 as m
    m.fa2_device_status(clear=True)
    return m


SCHEDULES = ("units", "balanced")


def run_gpu(fa2, q, k, v, w, out=None, lse=None, stream=None, schedule="balanced"):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    O, L = fa2.attention_forward(qd, kd, vd, scale=w.scale, is_causal=w.causal, out=out, lse=lse,
                                 stream=stream, schedule=schedule)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(clear=True) == 0, "device watchdog fired"
    return O, L


def compare(fa2, oracle_mod, w, rows=None, sample=None, schedule="balanced"):
    q, k, v = workloads.make_inputs(w)
    O, L = run_gpu(fa2, q, k, v, w, schedule=schedule)
    assert torch.isfinite(O).all().item(), "non-finite output"
    assert torch.isfinite(L).all().item(), "non-finite LSE"
    if sample is not None:
        rows = oracle_mod.sample_rows(w.B, w.H, w.N, sample, seed=w.seed)
    Oref, Lref = oracle_mod.attention_fwd(q, k, v, w.scale, w.causal, rows=rows)
    Og = O.float().cpu().numpy().astype(np.float64)
    Lg = L.cpu().numpy().astype(np.float64)
    if rows is not None:
        Og = Og.reshape(-1, w.D)[rows]
        Lg = Lg.reshape(-1)[rows]
    err_o = float(np.abs(Og - Oref).max())
    err_l = float(np.abs(Lg - Lref).max())
    assert err_o <= TOL_O[w.dtype], f"{w.describe()}: max|dO| = {err_o:.3e}"
    assert err_l <= TOL_LSE, f"{w.describe()}: max|dLSE| = {err_l:.3e}"
    return err_o, err_l


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_tiny_every_element(fa2, oracle_mod, schedule):
    compare(fa2, oracle_mod, workloads.WORKLOADS["tiny"], schedule=schedule)


EDGE_N = [1, 7, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 1000]


@pytest.mark.parametrize("N", EDGE_N)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("schedule", SCHEDULES)
def test_edge_shapes_every_element(fa2, oracle_mod, N, D, dtype, causal, schedule):
    w = workloads.custom(1, 2, N, D, dtype, causal, seed=N * 7 + D)
    compare(fa2, oracle_mod, w, schedule=schedule)


EDGE_N_PADDED = [1, 63, 129, 256, 257, 1000]


@pytest.mark.parametrize("N", EDGE_N_PADDED)
@pytest.mark.parametrize("D", [32, 96])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("schedule", SCHEDULES)
def test_padded_head_dims_every_element(fa2, oracle_mod, N, D, dtype, causal, schedule):
    # Head dims 32 and 96 run in the tiles of 64 and 128 with zero-filled
    # columns; a column past D read from memory (the next row's first
    # elements) instead of as zero would change every score of its row.
    w = workloads.custom(2, 3, N, D, dtype, causal, seed=N * 11 + D)
    compare(fa2, oracle_mod, w, schedule=schedule)


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("name", ["pages_d32", "target_d96", "target_d256"])
def test_other_head_dim_workloads_full_size(fa2, oracle_mod, name, schedule):
    compare(fa2, oracle_mod, workloads.WORKLOADS[name], sample=600, schedule=schedule)


EDGE_N_256 = [1, 63, 127, 128, 129, 255, 256, 257, 1000]


@pytest.mark.parametrize("N", EDGE_N_256)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("schedule", SCHEDULES)
def test_head_dim_256_every_element(fa2, oracle_mod, N, dtype, causal, schedule):
    # Head dim 256 runs on its own kernel: 128-row work units, two S buffers.
    w = workloads.custom(2, 3, N, 256, dtype, causal, seed=N * 13 + 256)
    compare(fa2, oracle_mod, w, schedule=schedule)


@pytest.mark.parametrize("shape", [(1, 1, 4096, False), (1, 2, 3000, True), (1, 3, 2049, False),
                                   (2, 1, 8192, False), (1, 1, 8192, True)])
def test_head_dim_256_units_cut_across_many_ctas(fa2, oracle_mod, shape):
    # Few K/V-tile steps per CTA at head dim 256: units split over several
    # CTAs, each owner merging several partials (every row checked).
    B, H, N, causal = shape
    w = workloads.custom(B, H, N, 256, "bf16", causal, seed=N + 256)
    compare(fa2, oracle_mod, w, schedule="balanced")


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_head_dim_256_many_units_per_cta(fa2, oracle_mod, schedule):
    w = workloads.custom(3, 50, 700, 256, "f16", True, seed=61)
    compare(fa2, oracle_mod, w, sample=400, schedule=schedule)
    w = workloads.custom(2, 90, 640, 256, "bf16", False, seed=62)
    compare(fa2, oracle_mod, w, sample=400, schedule=schedule)


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_head_dim_256_peaked_logits(fa2, oracle_mod, schedule):
    # Q/K ~ N(0, 3^2) as in the ragged workload: sharply peaked rows in fp16.
    w = workloads.custom(2, 2, 1000, 256, "f16", False, seed=63, sigma_qk=3.0)
    compare(fa2, oracle_mod, w, schedule=schedule)


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_ragged_tail_does_not_read_the_next_head(fa2, oracle_mod, schedule):
    # Rows past N of one head must read as zeros, never as the next head's rows.
    w = workloads.custom(2, 3, 65, 64, "f16", False, seed=99)
    compare(fa2, oracle_mod, w, schedule=schedule)
    w = workloads.custom(2, 3, 200, 128, "bf16", True, seed=98)
    compare(fa2, oracle_mod, w, schedule=schedule)


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_many_units_per_cta(fa2, oracle_mod, schedule):
    # More work units than SMs: each persistent CTA loops over several units.
    w = workloads.custom(4, 40, 512, 64, "bf16", False, seed=5)
    compare(fa2, oracle_mod, w, sample=400, schedule=schedule)
    w = workloads.custom(3, 50, 700, 128, "f16", True, seed=6)
    compare(fa2, oracle_mod, w, sample=400, schedule=schedule)


@pytest.mark.parametrize("shape", [(1, 1, 4096, 128, False), (1, 1, 4096, 64, True), (1, 2, 3000, 128, True),
                                   (1, 3, 2049, 64, False), (2, 1, 8192, 128, False)])
def test_units_cut_across_many_ctas(fa2, oracle_mod, shape):
    # Few K/V-tile steps per CTA: one query tile's K/V range is split over
    # several CTAs and its owner merges several partials (every row checked).
    B, H, N, D, causal = shape
    w = workloads.custom(B, H, N, D, "bf16", causal, seed=N + D)
    compare(fa2, oracle_mod, w, schedule="balanced")


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("name", workloads.CONTRACT + ("target", "target_f16"))
def test_contract_workloads_full_size(fa2, oracle_mod, name, schedule):
    w = workloads.WORKLOADS[name]
    if w.B * w.H * w.N <= 4096:
        compare(fa2, oracle_mod, w, schedule=schedule)
    else:
        compare(fa2, oracle_mod, w, sample=600, schedule=schedule)


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_peaked_logits_every_element(fa2, oracle_mod, schedule):
    # The ragged workload's Q/K ~ N(0, 3^2): sharply peaked rows, checked on every row.
    w = workloads.WORKLOADS["ragged"]
    compare(fa2, oracle_mod, workloads.custom(w.B, 2, w.N, w.D, w.dtype, w.causal, w.seed, sigma_qk=3.0),
            schedule=schedule)


def test_outputs_fully_overwritten_and_deterministic(fa2, oracle_mod):
    w = workloads.custom(2, 4, 300, 128, "bf16", True, seed=12)
    q, k, v = workloads.make_inputs(w)
    out = torch.full((w.B, w.H, w.N, w.D), float("nan"), dtype=w.torch_dtype, device="cuda")
    lse = torch.full((w.B, w.H, w.N), float("nan"), dtype=torch.float32, device="cuda")
    O1, L1 = run_gpu(fa2, q, k, v, w, out=out, lse=lse)
    assert O1.data_ptr() == out.data_ptr()
    assert torch.isfinite(O1).all().item() and torch.isfinite(L1).all().item()
    O2, L2 = run_gpu(fa2, q, k, v, w)
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
    O3, L3 = run_gpu(fa2, q, k, v, w, schedule="units")
    O4, L4 = run_gpu(fa2, q, k, v, w, schedule="units")
    assert torch.equal(O3, O4) and torch.equal(L3, L4)


def test_runs_on_a_side_stream(fa2, oracle_mod):
    w = workloads.custom(1, 3, 333, 64, "f16", True, seed=13)
    q, k, v = workloads.make_inputs(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        O, L = run_gpu(fa2, q, k, v, w, stream=s)
    Oref, Lref = oracle_mod.attention_fwd(q, k, v, w.scale, w.causal)
    assert np.abs(O.float().cpu().numpy() - Oref).max() <= TOL_O["f16"]
    assert np.abs(L.cpu().numpy() - Lref).max() <= TOL_LSE


def test_non_default_scale(fa2, oracle_mod):
    for scale in (0.01, 0.5):
        w = workloads.custom(1, 2, 257, 64, "bf16", False, seed=14)
        q, k, v = workloads.make_inputs(w)
        qd, kd, vd = (t.cuda() for t in (q, k, v))
        O, L = fa2.attention_forward(qd, kd, vd, scale=scale)
        torch.cuda.synchronize()
        Oref, Lref = oracle_mod.attention_fwd(q, k, v, scale, False)
        assert np.abs(O.float().cpu().numpy() - Oref).max() <= TOL_O["bf16"]
        assert np.abs(L.cpu().numpy() - Lref).max() <= TOL_LSE


def test_empty_problem(fa2):
    q = torch.empty(1, 2, 0, 64, dtype=torch.float16, device="cuda")
    O, L = fa2.attention_forward(q, q, q)
    torch.cuda.synchronize()
    assert O.shape == (1, 2, 0, 64) and L.shape == (1, 2, 0)
