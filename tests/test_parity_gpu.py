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
@pytest.mark.parametrize("name", ["pages_d32", "target_d96", "target_d256", "target_d512", "target_d1024"])
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


EDGE_N_DTILE = [1, 63, 128, 129, 255, 257, 700]


@pytest.mark.parametrize("N", EDGE_N_DTILE)
@pytest.mark.parametrize("D", [512, 1024])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_d_tiled_head_dims_every_element(fa2, oracle_mod, N, D, dtype, causal):
    # Head dims 512 and 1024: units of 128 query rows and one 256-column
    # chunk of O, each recomputing the full S over all of D; Q and K stream
    # through the ring in 128-column chunks, V in 64-key halves of the
    # unit's columns (round schedule only: "balanced" runs the rounds).
    w = workloads.custom(2, 2, N, D, dtype, causal, seed=N * 17 + D)
    compare(fa2, oracle_mod, w, schedule="units")


@pytest.mark.parametrize("D", [512, 1024])
def test_d_tiled_many_units_per_cta_and_balanced_request(fa2, oracle_mod, D):
    # More units than SMs (each CTA walks several (query tile, output chunk)
    # units, the ring and barriers carrying over); a balanced request runs the
    # rounds and gives the same output bit for bit.
    w = workloads.custom(2, 20, 1024, D, "bf16", False, seed=D + 5)
    q, k, v = workloads.make_inputs(w)
    O1, L1 = run_gpu(fa2, q, k, v, w, schedule="units")
    O2, L2 = run_gpu(fa2, q, k, v, w, schedule="balanced")
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
    compare(fa2, oracle_mod, w, sample=300, schedule="units")
    wc = workloads.custom(1, 12, 1500, D, "f16", True, seed=D + 6)
    compare(fa2, oracle_mod, wc, sample=300, schedule="units")


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


# ------------------------------------------------------- online-softmax corners
# Inputs drawn to reach the branches i.i.d. N(0, 1) scores never reach:
#   rising         the row maximum grows by ~17 (log2 units) per K/V tile, so
#                  the exponent base moves and O is rescaled in TMEM on almost
#                  every tile after a row's first (the correction step), and
#                  partial results cut between CTAs carry very different bases;
#   negative       every score is below -100 (natural log): a running max that
#                  started at 0 instead of -inf would underflow every weight
#                  (the CUDA book's -inf guard note, section 15.3);
#   dominant_last  one key in the last, ragged K/V tile outweighs the rest by
#                  ~20 nats: the base moves on the tile that is also masked
#                  past N (and on the causal diagonal).
LOG2E = 1.0 / np.log(2.0)
RESCALE_LOG2 = 8.0  # the kernel moves a row's exponent base when its max passes the base by more than this


def _scores(q, k, scale, causal):
    """fp64 scores [B*H, N, N] with disallowed keys at -inf (test-side, from the exact 16-bit inputs)."""
    qd = q.double().reshape(-1, q.shape[2], q.shape[3])
    kd = k.double().reshape(-1, k.shape[2], k.shape[3])
    s = torch.matmul(qd, kd.transpose(1, 2)) * scale
    if causal:
        n = s.shape[1]
        s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    return s.numpy()


def base_moves_after_first_tile(q, k, scale, causal, tile=128):
    """Per row: how many K/V tiles after its first allowed one move the exponent base, with the rule the
    kernel applies (running max in log2 units more than RESCALE_LOG2 above the base) and whole rows
    walked tile by tile (the round schedule)."""
    s = _scores(q, k, scale, causal) * LOG2E
    n = s.shape[2]
    run = np.full(s.shape[:2], -np.inf)
    base = np.full(s.shape[:2], -np.inf)
    moves = np.zeros(s.shape[:2], dtype=np.int64)
    for j0 in range(0, n, tile):
        run = np.maximum(run, s[:, :, j0:j0 + tile].max(axis=2))
        move = np.isfinite(run) & (~np.isfinite(base) | (run - base > RESCALE_LOG2))
        moves += (move & np.isfinite(base)).astype(np.int64)
        base = np.where(move, run, base)
    return moves


CORNER_D = [32, 64, 96, 128, 256, 512, 1024]


def lse_tolerance(q, k, w):
    """TOL_LSE plus the fp32 accumulation bound of the scores: the tensor core
    sums D/16 K-steps of 16 products into an fp32 accumulator, each step
    rounding it by at most one ulp (2^-23 relative) of a partial sum no larger
    than sum_d |q_d k_d|; the LSE, a smooth maximum of the scores, moves by at
    most the largest score error. Small for ordinary inputs (about 1e-5
    at D = 128 for N(0, 1) data); it matters only where every score has a
    huge raw magnitude (the all-negative inputs at D = 1024: sum |q k| ~ 5e3)."""
    qa = q.double().abs().reshape(-1, q.shape[2], q.shape[3])
    ka = k.double().abs().reshape(-1, k.shape[2], k.shape[3])
    l1 = float(torch.matmul(qa, ka.transpose(1, 2)).max())
    return TOL_LSE + w.scale * (w.D / 16) * 2.0 ** -23 * l1


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", CORNER_D)
@pytest.mark.parametrize("kind", workloads.STRUCTURED_KINDS)
def test_online_softmax_corners_every_element(fa2, oracle_mod, kind, D, dtype, causal, schedule):
    # B1 H2 N1000: on the balanced schedule the 32-64 K/V-tile steps of the
    # problem spread over as many CTAs, so every unit is cut and merged from
    # partials; on the round schedule each CTA walks whole rows of 8 tiles.
    w = workloads.custom(1, 2, 1000, D, dtype, causal, seed=D * 5 + len(kind))
    q, k, v = workloads.make_structured_inputs(w, kind)
    # the inputs reach the branch they are drawn for
    if kind == "rising":
        moves = base_moves_after_first_tile(q, k, w.scale, causal)
        assert (moves > 0).mean() > 0.8, "rising scores must move the exponent base after the first tile"
    elif kind == "negative":
        s = _scores(q, k, w.scale, causal)
        assert np.nanmax(np.where(np.isfinite(s), s, np.nan)) < -88.0, "every score must underflow exp()"
    else:
        js = workloads.dominant_key(w.N)
        moves = base_moves_after_first_tile(q, k, w.scale, causal)
        assert (moves[:, js:] > 0).mean() > 0.9, "the dominant key must move the base on the last tile"
    O, L = run_gpu(fa2, q, k, v, w, schedule=schedule)
    assert torch.isfinite(O).all().item() and torch.isfinite(L).all().item()
    Oref, Lref = oracle_mod.attention_fwd(q, k, v, w.scale, w.causal)
    err_o = float(np.abs(O.float().cpu().numpy() - Oref).max())
    err_l = float(np.abs(L.cpu().numpy() - Lref).max())
    tol_l = lse_tolerance(q, k, w)
    assert err_o <= TOL_O[dtype], f"{kind} {w.describe()} {schedule}: max|dO| = {err_o:.3e}"
    assert err_l <= tol_l, f"{kind} {w.describe()} {schedule}: max|dLSE| = {err_l:.3e} (bound {tol_l:.3e})"


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("shape", [(1, 2, 2049, 128, "bf16", False), (2, 3, 1537, 64, "f16", True),
                                   (1, 2, 2000, 256, "bf16", True), (3, 40, 700, 128, "f16", False)])
def test_rising_scores_longer_rows_and_many_units(fa2, oracle_mod, shape, schedule):
    # Longer rows (16-17 tiles whose base moves on each), and more units than
    # SMs (each CTA's later units start from a base left by an earlier one).
    B, H, N, D, dtype, causal = shape
    w = workloads.custom(B, H, N, D, dtype, causal, seed=N + D + 3)
    q, k, v = workloads.make_structured_inputs(w, "rising")
    O, L = run_gpu(fa2, q, k, v, w, schedule=schedule)
    rows = oracle_mod.sample_rows(B, H, N, 500, seed=w.seed) if B * H > 8 else None
    Oref, Lref = oracle_mod.attention_fwd(q, k, v, w.scale, w.causal, rows=rows)
    Og = O.float().cpu().numpy()
    Lg = L.cpu().numpy()
    if rows is not None:
        Og = Og.reshape(-1, D)[rows]
        Lg = Lg.reshape(-1)[rows]
    assert float(np.abs(Og - Oref).max()) <= TOL_O[dtype]
    assert float(np.abs(Lg - Lref).max()) <= TOL_LSE


@pytest.mark.parametrize("shape", [(1, 2, 4096, 128, False), (1, 38, 1024, 128, False), (1, 39, 1024, 128, False),
                                   (2, 3, 1000, 64, True), (1, 4, 2048, 256, False), (1, 2, 1500, 512, False)])
def test_auto_schedule_in_c_runs_the_named_schedule(fa2, shape):
    # fa2_fwd_sched(FA2_SCHED_AUTO) takes the schedule fa2_fwd_schedule_for
    # names: its output is bit-identical to that schedule's own entry point
    # (fa2_fwd_ws for balanced, fa2_fwd for the rounds).
    B, H, N, D, causal = shape
    w = workloads.custom(B, H, N, D, "bf16", causal, seed=B * H + N)
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    named = fa2.fa2_fwd_schedule_for(B, H, N, D, causal, sms)
    ws = torch.empty(fa2.fa2_fwd_workspace_bytes(D), dtype=torch.uint8, device="cuda")
    outs = []
    for entry in ("auto", "named"):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, D, w.scale,
                int(causal), fa2.FA2_BF16)
        s = torch.cuda.current_stream().cuda_stream
        if entry == "auto":
            rc = fa2.fa2_fwd_sched(*ptrs, ws.data_ptr(), ws.numel(), fa2.FA2_SCHED_AUTO, s)
        elif named == fa2.FA2_SCHED_BALANCED:
            rc = fa2.fa2_fwd_ws(*ptrs, ws.data_ptr(), ws.numel(), s)
        else:
            rc = fa2.fa2_fwd(*ptrs, s)
        assert rc == fa2.FA2_OK, fa2.error_text(rc)
        torch.cuda.synchronize()
        outs.append((o, lse))
    assert fa2.fa2_device_status(clear=True) == 0
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    # with no workspace the library's choice is always the rounds (fa2_fwd)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    rc = fa2.fa2_fwd_sched(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, D,
                           w.scale, int(causal), fa2.FA2_BF16, None, 0, fa2.FA2_SCHED_AUTO,
                           torch.cuda.current_stream().cuda_stream)
    assert rc == fa2.FA2_OK, fa2.error_text(rc)
    o_u = torch.empty_like(q)
    l_u = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    rc = fa2.fa2_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_u.data_ptr(), l_u.data_ptr(), B, H, N, D, w.scale,
                     int(causal), fa2.FA2_BF16, torch.cuda.current_stream().cuda_stream)
    assert rc == fa2.FA2_OK, fa2.error_text(rc)
    torch.cuda.synchronize()
    assert torch.equal(o, o_u) and torch.equal(lse, l_u)
