"""GB300 (sm_103a) FlashAttention-2 forward and backward: a C-ABI library plus a thin Python binding.

    from attention_forward_03_gb300 import attention_forward, attention_backward
    O, LSE = attention_forward(q, k, v, is_causal=True)
    dQ, dK, dV = attention_backward(q, k, v, O, LSE, dO, is_causal=True)

The compute runs in libfa2_gb300.so (build it with
``attention_forward_03_gb300.build.build()``); the binding fails loudly if it
is missing.
"""
from .binding import (  # noqa: F401
    FA2_BF16, FA2_ERR_ALIGN, FA2_ERR_CUDA, FA2_ERR_INVALID_ARG, FA2_ERR_TIMEOUT, FA2_ERR_UNSUPPORTED,
    FA2_F16, FA2_OK, FA2_SCHED_AUTO, FA2_SCHED_BALANCED, FA2_SCHED_UNITS, Fa2Error, attention_backward,
    attention_forward, attention_forward_host, error_text, fa2_bwd, fa2_bwd_sched, fa2_bwd_workspace_bytes,
    fa2_device_status, fa2_fwd, fa2_fwd_host_buffer_bytes, fa2_fwd_sched, fa2_fwd_schedule_for,
    fa2_fwd_workspace_bytes, fa2_fwd_ws, fa2_set_watchdog_ns, fa2_version, library, workspace_for,
)
