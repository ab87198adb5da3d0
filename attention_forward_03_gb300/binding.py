"""Thin ctypes binding over the C ABI in include/fa2.h (argument marshalling only).

Every step of the forward pass runs in the sm_103a kernels of
libfa2_gb300.so. This module only turns tensors into pointers, sizes and a
stream handle, and turns status codes into exceptions. There is no fallback:
if the library is missing, importing the functions below raises.
"""
from __future__ import annotations

import ctypes
import math
import os

LIB_NAME = "libfa2_gb300.so"
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), LIB_NAME)

FA2_F16 = 0
FA2_BF16 = 1
FA2_OK = 0
FA2_ERR_INVALID_ARG = -1
FA2_ERR_UNSUPPORTED = -2
FA2_ERR_ALIGN = -3
FA2_ERR_CUDA = -4
FA2_ERR_TIMEOUT = -5

# every symbol include/fa2.h declares, with its ctypes signature
_VP = ctypes.c_void_p
SIGNATURES = {
    "fa2_fwd": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int, _VP]),
    "fa2_fwd_workspace_bytes": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "fa2_fwd_ws": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int, _VP, ctypes.c_size_t,
                                  _VP]),
    "fa2_fwd_noalloc": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int, _VP]),
    "fa2_device_status": (ctypes.c_int, [_VP, ctypes.POINTER(ctypes.c_int), ctypes.c_int]),
    "fa2_set_watchdog_ns": (ctypes.c_int, [ctypes.c_ulonglong]),
    "fa2_test_withhold_next_load": (ctypes.c_int, [ctypes.c_int]),
    "fa2_error_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fa2_last_cuda_error": (ctypes.c_char_p, []),
    "fa2_version": (ctypes.c_int, []),
}

_lib = None


class Fa2Error(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(what)
        self.code = code


def library() -> ctypes.CDLL:
    """Load libfa2_gb300.so (built in-tree by attention_forward_03_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_NAME} is not built (expected at {LIB_PATH}); "
                              "run attention_forward_03_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def error_text(code: int) -> str:
    lib = library()
    msg = lib.fa2_error_string(code).decode()
    if code == FA2_ERR_CUDA:
        msg += f" ({lib.fa2_last_cuda_error().decode()})"
    return msg


def _check(code: int, what: str) -> None:
    if code != FA2_OK:
        raise Fa2Error(code, f"{what}: {error_text(code)} [{code}]")


def fa2_fwd(Q: int, K: int, V: int, O: int, LSE: int, B: int, H: int, N: int, D: int, scale: float,
            is_causal: int, dtype: int, stream: int | None) -> int:
    """Pointer-level call with the C ABI's argument list; returns the raw status code."""
    return library().fa2_fwd(Q, K, V, O, LSE, B, H, N, D, float(scale), int(is_causal), int(dtype), stream)


def fa2_fwd_ws(Q: int, K: int, V: int, O: int, LSE: int, B: int, H: int, N: int, D: int, scale: float,
               is_causal: int, dtype: int, workspace: int | None, workspace_bytes: int, stream: int | None) -> int:
    """Pointer-level call of the workspace variant; returns the raw status code."""
    return library().fa2_fwd_ws(Q, K, V, O, LSE, B, H, N, D, float(scale), int(is_causal), int(dtype), workspace,
                                int(workspace_bytes), stream)


def fa2_fwd_workspace_bytes(D: int) -> int:
    n = ctypes.c_size_t(0)
    _check(library().fa2_fwd_workspace_bytes(int(D), ctypes.byref(n)), "fa2_fwd_workspace_bytes")
    return n.value


def fa2_device_status(stream: int | None = None, clear: bool = False) -> int:
    v = ctypes.c_int(0)
    _check(library().fa2_device_status(stream, ctypes.byref(v), int(bool(clear))), "fa2_device_status")
    return v.value


def fa2_set_watchdog_ns(ns: int) -> None:
    _check(library().fa2_set_watchdog_ns(int(ns)), "fa2_set_watchdog_ns")


def fa2_version() -> int:
    return library().fa2_version()


# ------------------------------------------------------------ tensor helpers
def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return FA2_F16
    if t.dtype == torch.bfloat16:
        return FA2_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; expected float16 or bfloat16")


_workspaces = {}


def workspace_for(device, D: int):
    """A cached caller-side workspace (torch uint8 tensor) for fa2_fwd_ws on `device`."""
    import torch
    dev = torch.device(device)
    key = (dev.index, D)
    ws = _workspaces.get(key)
    if ws is None:
        with torch.cuda.device(dev):
            n = fa2_fwd_workspace_bytes(D)
        ws = torch.empty(n, dtype=torch.uint8, device=dev)
        _workspaces[key] = ws
    return ws


UNIT_ROWS = 256  # query rows per work unit of the kernel


def choose_schedule(B: int, H: int, N: int, is_causal: bool, sms: int) -> str:
    """Pick the kernel schedule for a problem (a choice between two C entry points).

    The balanced schedule (fa2_fwd_ws) splits work exactly across the SMs at the
    cost of a partial-result merge per CTA; it pays off only for non-causal work
    of at least one unit per SM whose last round of whole units would leave more
    than 8% of the SMs idle. Causal work is already balanced by the round
    schedule's heaviest-first zig-zag, and small problems are dominated by the
    fixed per-segment cost, so both use the round schedule (fa2_fwd).
    """
    units = B * H * -(-N // UNIT_ROWS)
    if is_causal or units < sms:
        return "units"
    rounds = -(-units // sms)
    return "balanced" if units / (rounds * sms) < 0.92 else "units"


def attention_forward(q, k, v, scale: float | None = None, is_causal: bool = False, out=None, lse=None,
                      stream=None, schedule: str = "auto", workspace=None):
    """FlashAttention-2 forward over torch CUDA tensors [B, H, N, D] (fp16/bf16).

    Returns (O, LSE): O like q, LSE float32 [B, H, N]. `out` / `lse` may be
    passed to write into caller-owned buffers. Runs on `stream` (a
    torch.cuda.Stream) or the current stream.
    schedule: "auto" (choose_schedule), "balanced" (fa2_fwd_ws with a
    workspace: equal work per SM) or "units" (fa2_fwd: whole query tiles per
    CTA, no workspace).
    workspace: optional uint8 CUDA tensor for the balanced schedule; by default
    a cached one per device is used.
    """
    import torch
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if q.shape != k.shape or q.shape != v.shape or q.dim() != 4:
        raise ValueError("q, k, v must share one [B, H, N, D] shape")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError("q, k, v must share one dtype")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    if schedule not in ("auto", "balanced", "units"):
        raise ValueError("schedule must be 'auto', 'balanced' or 'units'")
    B, H, N, D = q.shape
    if schedule == "auto":
        sms = torch.cuda.get_device_properties(q.device).multi_processor_count
        schedule = choose_schedule(B, H, N, is_causal, sms)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like q")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        if schedule == "units":
            code = fa2_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                           B, H, N, D, scale, int(bool(is_causal)), _dtype_code(q), s.cuda_stream)
            _check(code, "fa2_fwd")
        else:
            ws = workspace if workspace is not None else workspace_for(q.device, D)
            code = fa2_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                              B, H, N, D, scale, int(bool(is_causal)), _dtype_code(q), ws.data_ptr(),
                              ws.numel() * ws.element_size(), s.cuda_stream)
            _check(code, "fa2_fwd_ws")
    return out, lse
