"""The scratch-free entry point fa2_fwd_noalloc, called through the C ABI.

It serves callers that may not allocate device memory (their application
owns all device memory through a fixed pool, or an allocation's latency and
implied synchronisation are not acceptable on their path). Its results must
match fa2_fwd_ws — the same schedule with caller-provided scratch — and stay
right on a second call, which reuses the static scratch the first call left
behind. This file is collected last so a stop-at-first-failure run has run
every other test first; it also passes on its own in a fresh process.
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
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from attention_forward_03_gb300 import build
    build.build()
    from attention_forward_03_gb300 import binding
    return binding


def _ptrs(*ts):
    return [t.data_ptr() for t in ts]


@pytest.mark.parametrize("shape", [(1, 8, 2048, 128, "bf16", False), (2, 3, 1000, 64, "f16", True),
                                   (1, 2, 3000, 128, "f16", True), (1, 3, 777, 96, "bf16", False),
                                   (1, 4, 1500, 256, "f16", True)])
def test_no_alloc_matches_the_workspace_entry_point(lib, shape):
    B, H, N, D, dtype, causal = shape
    w = workloads.custom(B, H, N, D, dtype, causal, seed=N + 7)
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    code = lib.FA2_BF16 if dtype == "bf16" else lib.FA2_F16
    stream = torch.cuda.current_stream().cuda_stream
    so = lib.library()

    ws = torch.empty(lib.fa2_fwd_workspace_bytes(D), dtype=torch.uint8, device="cuda")
    o_ref = torch.empty_like(q)
    l_ref = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    rc = so.fa2_fwd_ws(*_ptrs(q, k, v, o_ref, l_ref), B, H, N, D, w.scale, int(causal), code,
                       ws.data_ptr(), ws.numel(), stream)
    assert rc == lib.FA2_OK, lib.error_text(rc)
    torch.cuda.synchronize()

    for call in range(2):  # the second call runs over the scratch the first one left
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        rc = so.fa2_fwd_noalloc(*_ptrs(q, k, v, o, lse), B, H, N, D, w.scale, int(causal), code, stream)
        assert rc == lib.FA2_OK, lib.error_text(rc)
        torch.cuda.synchronize()
        assert lib.fa2_device_status(clear=True) == 0
        err_o = float((o.float() - o_ref.float()).abs().max())
        err_l = float((lse - l_ref).abs().max())
        assert np.isfinite(err_o) and err_o <= TOL_O[dtype], f"call {call}: max|dO| = {err_o}"
        assert np.isfinite(err_l) and err_l <= TOL_LSE, f"call {call}: max|dLSE| = {err_l}"
