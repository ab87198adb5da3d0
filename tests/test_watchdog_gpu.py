"""The device watchdog, exercised without any GPU fault.

A test hook makes the next launch withhold its first K/V tile, so the waits
for it run out after a short watchdog time. The kernel must record the wait
site in the status word, wind down, and leave the context usable: a normal
launch right after must still match the oracle.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa2():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from attention_forward_03_gb300 import build
    build.build()
    import attention_forward_03_gb300 as m
    m.fa2_device_status(clear=True)
    return m


@pytest.mark.parametrize("D", [128, 256, 512])
def test_withheld_tile_times_out_and_the_context_stays_usable(fa2, oracle_mod, D):
    w = workloads.custom(1, 4, 512, D, "bf16", False, seed=77)
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    lib = fa2.library()
    try:
        fa2.fa2_set_watchdog_ns(20_000_000)  # 20 ms
        assert lib.fa2_test_withhold_next_load(1) == fa2.FA2_OK
        fa2.attention_forward(q, k, v, scale=w.scale, schedule="units")
        torch.cuda.synchronize()  # returns: every wait in the kernel is bounded
        # the C call reports the timeout as FA2_ERR_TIMEOUT, with the wait site in the word
        site = ctypes.c_int(0)
        assert lib.fa2_device_status(None, ctypes.byref(site), 0) == fa2.FA2_ERR_TIMEOUT
        assert site.value > 0
        status = fa2.fa2_device_status(clear=True)
        assert status == site.value, "the withheld tile should have made a wait run out"
        assert fa2.fa2_device_status() == 0  # cleared
        assert lib.fa2_device_status(None, ctypes.byref(site), 0) == fa2.FA2_OK and site.value == 0
    finally:
        lib.fa2_test_withhold_next_load(0)
        fa2.fa2_set_watchdog_ns(0)
    # the hook applied to one launch only; the next one is normal and right
    O, L = fa2.attention_forward(q, k, v, scale=w.scale, schedule="units")
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(clear=True) == 0
    Oref, Lref = oracle_mod.attention_fwd(q.cpu(), k.cpu(), v.cpu(), w.scale, False)
    assert np.abs(O.float().cpu().numpy() - Oref).max() <= 1e-2
    assert np.abs(L.cpu().numpy() - Lref).max() <= 1e-3


@pytest.mark.parametrize("D,schedule", [(128, "units"), (128, "balanced"), (64, "balanced")])
def test_backward_withheld_tile_times_out_and_the_context_stays_usable(fa2, oracle_mod, D, schedule):
    # The backward's main kernel takes the hook: its first K/V tile never
    # arrives, every wait on it runs out, the balanced schedule's cross-CTA
    # waits end too, and a normal call right after is right.
    w = workloads.custom(1, 3, 640, D, "bf16", False, seed=78)
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    do = workloads.make_grad_output(w).cuda()
    O, L = fa2.attention_forward(q, k, v, scale=w.scale)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(clear=True) == 0
    lib = fa2.library()
    try:
        fa2.fa2_set_watchdog_ns(20_000_000)  # 20 ms
        assert lib.fa2_test_withhold_next_load(1) == fa2.FA2_OK
        fa2.attention_backward(q, k, v, O, L, do, scale=w.scale, schedule=schedule)
        torch.cuda.synchronize()  # returns: every wait in the kernel is bounded
        assert fa2.fa2_device_status(clear=True) != 0, "the withheld tile should have made a wait run out"
    finally:
        lib.fa2_test_withhold_next_load(0)
        fa2.fa2_set_watchdog_ns(0)
    dq, dk, dv = fa2.attention_backward(q, k, v, O, L, do, scale=w.scale, schedule=schedule)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(clear=True) == 0
    ref = oracle_mod.attention_bwd(q.cpu(), k.cpu(), v.cpu(), do.cpu(), w.scale, False, magnitudes=True)
    u = 2.0 ** -8
    for name, g in zip(("dq", "dk", "dv"), (dq, dk, dv)):
        r, m = ref[name], ref[name + "_mag"]
        bound = 3 * u * m + u * np.abs(r) + 2.0 ** -20 * m.max()
        assert float((np.abs(g.float().cpu().numpy() - r) / bound).max()) <= 1.0, name

