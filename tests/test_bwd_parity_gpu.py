"""Parity of the sm_103a backward pass with the CPU fp64 gradient oracle, through the C ABI.

Inputs: the seeded Q, K, V of a workload and an upstream gradient dO
(workloads.make_grad_output). The GPU runs its own forward (fa2_fwd: O and
LSE) and then fa2_bwd; the oracle differentiates the exact definition.

Tolerance, per element x of dQ, dK and dV (derived from the arithmetic):
  |x_gpu - x_ref| <= 3u * cond(x) + u * |x_ref| + 2^-20 * max(cond)
with u the unit roundoff of the dtype (2^-11 fp16, 2^-8 bf16) and cond(x)
the oracle's condition sum: a relative change u of every P, dS and O value,
which the kernel rounds to the dtype before the tensor core reads them, moves
x by at most about u * cond(x). The factor 3 covers those three roundings;
u * |x_ref| is the rounding of the output; the last term covers fp32
accumulation (ex2.approx, MMA and atomic summation order), far below u.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

U = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}


@pytest.fixture(scope="module")
def fa2():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from attention_forward_03_gb300 import build
    build.build()
    import attention_forward_03_gb300 as m
    m.fa2_device_status(clear=True)
    return m


def run_gpu(fa2, w, q, k, v, do, stream=None, outs=None, workspace=None, schedule="auto"):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    O, L = fa2.attention_forward(qd, kd, vd, scale=w.scale, is_causal=w.causal)
    kw = {}
    if outs is not None:
        kw = dict(dq=outs[0], dk=outs[1], dv=outs[2])
    grads = fa2.attention_backward(qd, kd, vd, O, L, dod, scale=w.scale, is_causal=w.causal, stream=stream,
                                   workspace=workspace, schedule=schedule, **kw)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(clear=True) == 0, "device watchdog fired"
    return dict(zip(("dq", "dk", "dv"), grads))


def check(w, gpu, ref, heads=None):
    """Compare GPU gradients (all heads, or the listed flat head ids) with the oracle's."""
    u = U[w.dtype]
    worst = {}
    for name in ("dq", "dk", "dv"):
        g = gpu[name].float().cpu().numpy().astype(np.float64).reshape(w.B * w.H, w.N, w.D)
        if heads is not None:
            g = g[np.asarray(heads)]
        r = ref[name].reshape(g.shape)
        m = ref[name + "_mag"].reshape(g.shape)
        assert np.isfinite(g).all(), f"{w.describe()} {name}: non-finite values"
        bound = 3 * u * m + u * np.abs(r) + 2.0 ** -20 * m.max()
        ratio = float((np.abs(g - r) / bound).max())
        worst[name] = (ratio, float(np.abs(g - r).max()))
        assert ratio <= 1.0, f"{w.describe()} {name}: error/bound = {ratio:.3f}, max|err| = {worst[name][1]:.3e}"
    return worst


def compare(fa2, oracle_mod, w, heads=None, schedule="auto"):
    q, k, v = workloads.make_inputs(w)
    do = workloads.make_grad_output(w)
    gpu = run_gpu(fa2, w, q, k, v, do, schedule=schedule)
    ref = oracle_mod.attention_bwd(q, k, v, do, w.scale, w.causal, heads=heads, magnitudes=True)
    return check(w, gpu, ref, heads)


def test_tiny_every_element(fa2, oracle_mod):
    compare(fa2, oracle_mod, workloads.WORKLOADS["tiny"])


EDGE_N = [1, 7, 63, 64, 65, 127, 128, 129, 255, 257, 1000]


SCHEDULES = ("units", "balanced")


@pytest.mark.parametrize("N", EDGE_N)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("schedule", SCHEDULES)
def test_edge_shapes_every_element(fa2, oracle_mod, N, D, dtype, causal, schedule):
    compare(fa2, oracle_mod, workloads.custom(1, 2, N, D, dtype, causal, seed=N * 11 + D), schedule=schedule)


EDGE_N_PADDED = [1, 63, 129, 257, 1000]


@pytest.mark.parametrize("N", EDGE_N_PADDED)
@pytest.mark.parametrize("D", [32, 96])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("schedule", SCHEDULES)
def test_padded_head_dims_every_element(fa2, oracle_mod, N, D, dtype, causal, schedule):
    """Head dims 32 and 96 run in the tiles of 64 and 128 with zero-filled columns."""
    compare(fa2, oracle_mod, workloads.custom(2, 2, N, D, dtype, causal, seed=N * 13 + D), schedule=schedule)


@pytest.mark.parametrize("D", [32, 96])
@pytest.mark.parametrize("causal", [False, True])
def test_padded_head_dims_long_rows(fa2, oracle_mod, D, causal):
    """Many query steps per K/V tile and several tiles per CTA, auto schedule."""
    compare(fa2, oracle_mod, workloads.custom(1, 3, 2500, D, "bf16", causal, seed=D + 90))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("schedule", SCHEDULES)
def test_many_units_per_cta(fa2, oracle_mod, causal, schedule):
    """160 K/V tiles on at most 152 CTAs: units after the first reuse TMEM, the ring and barriers."""
    compare(fa2, oracle_mod, workloads.custom(1, 40, 512, 64, "bf16", causal, seed=77), schedule=schedule)


@pytest.mark.parametrize("shape", [(1, 1, 4096, 128, False), (1, 2, 3000, 128, True), (1, 3, 2049, 64, False),
                                   (2, 1, 8192, 64, True), (1, 1, 700, 128, False)])
def test_units_cut_across_many_ctas(fa2, oracle_mod, shape):
    """Balanced schedule with few query steps per CTA: one K/V tile's steps are split over several CTAs
    and its owner adds several partial dK, dV (every element checked)."""
    B, H, N, D, causal = shape
    compare(fa2, oracle_mod, workloads.custom(B, H, N, D, "bf16", causal, seed=N + D + 5), schedule="balanced")


@pytest.mark.parametrize("D", [64, 128])
def test_long_rows_every_element(fa2, oracle_mod, D):
    """Many query steps per unit (N = 2048: 32 steps of 64 rows) and ragged N."""
    compare(fa2, oracle_mod, workloads.custom(1, 2, 2000, D, "f16", True, seed=78))


def test_peaked_logits_every_element(fa2, oracle_mod):
    """Q, K ~ N(0, 3^2): sharply peaked rows, P close to one-hot."""
    compare(fa2, oracle_mod, workloads.custom(2, 3, 700, 64, "f16", False, seed=79, sigma_qk=3.0))


@pytest.mark.parametrize("name", workloads.CONTRACT + ("target",))
def test_contract_workloads_full_size(fa2, oracle_mod, name):
    """Full-size workloads, launched as the benchmark launches them; the oracle checks the
    first and last head whole (every row of dQ, dK and dV there)."""
    w = workloads.WORKLOADS[name]
    heads = [w.B * w.H - 1] if w.N > 16384 else [0, w.B * w.H - 1]
    compare(fa2, oracle_mod, w, heads=heads)


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_workspace_and_outputs_may_hold_garbage(fa2, oracle_mod, schedule):
    """The workspace (fp32 accumulator, row statistics, partial slots and flags) and the outputs start
    as NaN bytes: every output element is written, the accumulator is cleared by the call itself and
    no stale flag is taken for a partial of this call."""
    w = workloads.custom(1, 3, 333, 128, "bf16", True, seed=80)
    q, k, v = workloads.make_inputs(w)
    do = workloads.make_grad_output(w)
    need = fa2.fa2_bwd_workspace_bytes(w.B, w.H, w.N, w.D)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    outs = [torch.full(q.shape, float("nan"), dtype=q.dtype, device="cuda") for _ in range(3)]
    ref = oracle_mod.attention_bwd(q, k, v, do, w.scale, w.causal, magnitudes=True)
    first = run_gpu(fa2, w, q, k, v, do, outs=outs, workspace=ws, schedule=schedule)
    check(w, first, ref)
    keep = {n: t.clone() for n, t in first.items()}
    second = run_gpu(fa2, w, q, k, v, do, outs=outs, workspace=ws, schedule=schedule)
    check(w, second, ref)
    # dK and dV are summed in one fixed order; dQ by atomics (order may vary)
    assert torch.equal(keep["dk"], second["dk"]) and torch.equal(keep["dv"], second["dv"])


def test_runs_on_a_side_stream(fa2, oracle_mod):
    w = workloads.custom(2, 2, 300, 64, "f16", False, seed=81)
    q, k, v = workloads.make_inputs(w)
    do = workloads.make_grad_output(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gpu = run_gpu(fa2, w, q, k, v, do, stream=s)
    ref = oracle_mod.attention_bwd(q, k, v, do, w.scale, w.causal, magnitudes=True)
    check(w, gpu, ref)


def test_non_default_scale(fa2, oracle_mod):
    w = workloads.custom(1, 2, 200, 128, "bf16", True, seed=82)
    q, k, v = workloads.make_inputs(w)
    do = workloads.make_grad_output(w)
    scale = 0.3
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    O, L = fa2.attention_forward(qd, kd, vd, scale=scale, is_causal=True)
    dq, dk, dv = fa2.attention_backward(qd, kd, vd, O, L, dod, scale=scale, is_causal=True)
    torch.cuda.synchronize()
    ref = oracle_mod.attention_bwd(q, k, v, do, scale, True, magnitudes=True)
    check(w, dict(dq=dq, dk=dk, dv=dv), ref)


def test_empty_problem(fa2):
    q = torch.empty(0, 2, 64, 64, dtype=torch.float16, device="cuda")
    lse = torch.empty(0, 2, 64, dtype=torch.float32, device="cuda")
    dq, dk, dv = fa2.attention_backward(q, q, q, q, lse, q)
    assert dq.numel() == 0 and dk.numel() == 0 and dv.numel() == 0


# Inputs drawn to reach the corners of the recomputed softmax (workloads.
# make_structured_inputs): "rising" scores grow by ~12 nats per K/V tile, so
# the forward's exponent base moves on almost every tile and P spans hundreds
# of orders of magnitude along a row; "dominant_last" puts one key that
# outweighs the rest by ~20 nats in the last, ragged K/V tile (and, causal, on
# the diagonal), so P is close to one-hot there.
@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [32, 64, 96, 128])
@pytest.mark.parametrize("kind", ["rising", "dominant_last"])
def test_softmax_corners_every_element(fa2, oracle_mod, kind, D, dtype, causal, schedule):
    w = workloads.custom(1, 2, 1000, D, dtype, causal, seed=D * 7 + len(kind))
    q, k, v = workloads.make_structured_inputs(w, kind)
    do = workloads.make_grad_output(w)
    gpu = run_gpu(fa2, w, q, k, v, do, schedule=schedule)
    ref = oracle_mod.attention_bwd(q, k, v, do, w.scale, w.causal, magnitudes=True)
    check(w, gpu, ref)
