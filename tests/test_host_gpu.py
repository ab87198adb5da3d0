"""fa2_fwd_host — the forward pass from and to host memory, pipelined in
chunks of heads — against the CPU fp64 oracle, and against the device-pointer
entry point, through the C ABI.

Tolerances as the device-path parity tests: O within 2e-3 (fp16) / 1e-2
(bf16), LSE within 1e-3 (max-abs against the oracle). With the round schedule
("units") every query tile is computed by one CTA in the same tile order
whichever launch it belongs to, so chunked results must equal the one-launch
results bit for bit.
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


def check_against_oracle(oracle_mod, w, q, k, v, O, L, rows=None):
    Oref, Lref = oracle_mod.attention_fwd(q, k, v, w.scale, w.causal, rows=rows)
    Og = O.float().numpy().astype(np.float64)
    Lg = L.numpy().astype(np.float64)
    if rows is not None:
        Og = Og.reshape(-1, w.D)[rows]
        Lg = Lg.reshape(-1)[rows]
    err_o = float(np.abs(Og - Oref).max())
    err_l = float(np.abs(Lg - Lref).max())
    assert err_o <= TOL_O[w.dtype], f"{w.describe()}: max|dO| = {err_o:.3e}"
    assert err_l <= TOL_LSE, f"{w.describe()}: max|dLSE| = {err_l:.3e}"


@pytest.mark.parametrize("heads_per_chunk", [1, 4, 6, None])
@pytest.mark.parametrize("schedule", ["units", "balanced"])
def test_chunked_host_path_matches_oracle(fa2, oracle_mod, heads_per_chunk, schedule):
    # 6 heads: chunks of 1, 4 (+ a ragged 2), all 6, and the default split
    w = workloads.custom(2, 3, 300, 64, "f16", False, seed=41)
    q, k, v = (t.pin_memory() for t in workloads.make_inputs(w))
    O, L = fa2.attention_forward_host(q, k, v, scale=w.scale, heads_per_chunk=heads_per_chunk, schedule=schedule)
    assert fa2.fa2_device_status(clear=True) == 0
    check_against_oracle(oracle_mod, w, q, k, v, O, L)


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "f16"), (96, "bf16"), (32, "f16"), (256, "bf16")])
def test_causal_host_path_matches_oracle(fa2, oracle_mod, D, dtype):
    w = workloads.custom(1, 5, 520, D, dtype, True, seed=42)
    q, k, v = (t.pin_memory() for t in workloads.make_inputs(w))
    O, L = fa2.attention_forward_host(q, k, v, scale=w.scale, is_causal=True, heads_per_chunk=2)
    assert fa2.fa2_device_status(clear=True) == 0
    check_against_oracle(oracle_mod, w, q, k, v, O, L)


def test_round_schedule_equals_device_entry_point_bit_for_bit(fa2):
    w = workloads.custom(2, 4, 700, 128, "bf16", False, seed=43)
    q, k, v = workloads.make_inputs(w)
    Od, Ld = fa2.attention_forward(q.cuda(), k.cuda(), v.cuda(), scale=w.scale, schedule="units")
    torch.cuda.synchronize()
    for hpc in (1, 3, 8):
        O, L = fa2.attention_forward_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), scale=w.scale,
                                          heads_per_chunk=hpc, schedule="units")
        assert torch.equal(O, Od.cpu()) and torch.equal(L, Ld.cpu()), f"heads_per_chunk={hpc}"


@pytest.mark.parametrize("N", [300, 301])
def test_packed_qkv_and_direct_lse_equal_the_copy_path(fa2, oracle_mod, N):
    # Q, K, V as slices of one page-locked [3, B, H, N, D] buffer take one 2-D
    # copy per chunk; page-locked LSE with N % 4 == 0 is written by the
    # kernels in place. The reference run uses unequally spaced inputs (slices
    # 0, 1 and 3 of a 4-slice buffer) and pageable LSE, the copy path. Same
    # kernels on the same chunks: equal bit for bit.
    w = workloads.custom(2, 3, N, 128, "bf16", False, seed=45)
    q, k, v = workloads.make_inputs(w)
    packed = torch.empty((3, *q.shape), dtype=q.dtype).pin_memory()
    spread = torch.empty((4, *q.shape), dtype=q.dtype).pin_memory()
    for i, t in enumerate((q, k, v)):
        packed[i].copy_(t)
        spread[(0, 1, 3)[i]].copy_(t)
    for hpc in (1, 2, None):
        lse_pinned = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
        O1, L1 = fa2.attention_forward_host(packed[0], packed[1], packed[2], scale=w.scale, lse=lse_pinned,
                                            heads_per_chunk=hpc, schedule="units")
        lse_pageable = torch.empty((w.B, w.H, w.N), dtype=torch.float32)
        O2, L2 = fa2.attention_forward_host(spread[0], spread[1], spread[3], scale=w.scale, lse=lse_pageable,
                                            heads_per_chunk=hpc, schedule="units")
        assert fa2.fa2_device_status(clear=True) == 0
        assert torch.equal(O1, O2) and torch.equal(L1, L2), f"heads_per_chunk={hpc}"
    check_against_oracle(oracle_mod, w, q, k, v, O1, L1)


def test_pageable_host_memory_and_side_stream(fa2, oracle_mod):
    w = workloads.custom(1, 3, 257, 64, "bf16", False, seed=44)
    q, k, v = workloads.make_inputs(w)  # pageable
    s = torch.cuda.Stream()
    out = torch.full(q.shape, float("nan"), dtype=q.dtype)
    lse = torch.full((w.B, w.H, w.N), float("nan"), dtype=torch.float32)
    O, L = fa2.attention_forward_host(q, k, v, scale=w.scale, out=out, lse=lse, stream=s, heads_per_chunk=1,
                                      synchronize=False)
    s.synchronize()
    assert O.data_ptr() == out.data_ptr() and L.data_ptr() == lse.data_ptr()
    check_against_oracle(oracle_mod, w, q, k, v, O, L)


def test_bench_workload_through_the_host_path(fa2, oracle_mod):
    # the end-to-end leg of the benchmark: the target workload with the
    # default chunking and schedule, checked on sampled rows
    w = workloads.WORKLOADS["target"]
    q, k, v = (t.pin_memory() for t in workloads.make_inputs(w))
    O, L = fa2.attention_forward_host(q, k, v, scale=w.scale, is_causal=w.causal)
    assert fa2.fa2_device_status(clear=True) == 0
    rows = oracle_mod.sample_rows(w.B, w.H, w.N, 400, seed=w.seed)
    check_against_oracle(oracle_mod, w, q, k, v, O, L, rows=rows)


def test_host_path_rejects_device_tensors_and_small_buffers(fa2):
    q = torch.zeros(1, 1, 64, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        fa2.attention_forward_host(q.cuda(), q.cuda(), q.cuda())
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        fa2.attention_forward_host(q, q, q, device_buffer=small)
    need = fa2.fa2_fwd_host_buffer_bytes(1, 1, 64, 64)
    big = torch.empty(need, dtype=torch.uint8, device="cuda")
    code = fa2.library().fa2_fwd_host(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), 1, 1,
                                      64, 64, 0.125, 0, 0, 0, 0, big.data_ptr(), need - 256, None)
    assert code == fa2.FA2_ERR_INVALID_ARG  # O overlaps the inputs
    out = torch.empty_like(q)
    lse = torch.empty(1, 1, 64)
    code = fa2.library().fa2_fwd_host(q.data_ptr(), q.data_ptr(), q.data_ptr(), out.data_ptr(), lse.data_ptr(), 1,
                                      1, 64, 64, 0.125, 0, 0, 0, 0, big.data_ptr(), need - 256, None)
    assert code == fa2.FA2_ERR_INVALID_ARG  # buffer too small
    code = fa2.library().fa2_fwd_host(q.data_ptr(), q.data_ptr(), q.data_ptr(), out.data_ptr(), lse.data_ptr(), 1,
                                      1, 64, 64, 0.125, 0, 0, 0, 0, big.data_ptr() + 16, need - 256, None)
    assert code == fa2.FA2_ERR_ALIGN
