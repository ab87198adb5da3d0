"""Thin ctypes binding over the C ABI in include/fa2.h (argument marshalling only).

Every step of the forward and backward passes runs in the sm_103a kernels of
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
FA2_SCHED_AUTO = 0
FA2_SCHED_UNITS = 1
FA2_SCHED_BALANCED = 2
_SCHEDULES = {"auto": FA2_SCHED_AUTO, "units": FA2_SCHED_UNITS, "balanced": FA2_SCHED_BALANCED}

# every symbol include/fa2.h declares, with its ctypes signature
_VP = ctypes.c_void_p
SIGNATURES = {
    "fa2_fwd": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int, _VP]),
    "fa2_fwd_workspace_bytes": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "fa2_fwd_ws": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int, _VP, ctypes.c_size_t,
                                  _VP]),
    "fa2_fwd_sched": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int, _VP, ctypes.c_size_t,
                                     ctypes.c_int, _VP]),
    "fa2_fwd_schedule_for": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.POINTER(ctypes.c_int)]),
    "fa2_fwd_noalloc": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int, _VP]),
    "fa2_fwd_host_buffer_bytes": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 ctypes.POINTER(ctypes.c_size_t)]),
    "fa2_fwd_host": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, _VP, ctypes.c_size_t, _VP]),
    "fa2_bwd_workspace_bytes": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.POINTER(ctypes.c_size_t)]),
    "fa2_bwd": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int,
                               ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int, _VP,
                               ctypes.c_size_t, _VP]),
    "fa2_bwd_sched": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int, _VP,
                                     ctypes.c_size_t, ctypes.c_int, _VP]),
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


def fa2_fwd_sched(Q: int, K: int, V: int, O: int, LSE: int, B: int, H: int, N: int, D: int, scale: float,
                  is_causal: int, dtype: int, workspace: int | None, workspace_bytes: int, schedule: int,
                  stream: int | None) -> int:
    """Pointer-level call with an explicit schedule code (FA2_SCHED_*); returns the raw status code."""
    return library().fa2_fwd_sched(Q, K, V, O, LSE, B, H, N, D, float(scale), int(is_causal), int(dtype), workspace,
                                   int(workspace_bytes), int(schedule), stream)


def fa2_fwd_schedule_for(B: int, H: int, N: int, D: int, is_causal: bool, sms: int) -> int:
    """The schedule code FA2_SCHED_AUTO takes for this problem on a device with `sms` SMs (host arithmetic)."""
    out = ctypes.c_int(0)
    _check(library().fa2_fwd_schedule_for(int(B), int(H), int(N), int(D), int(bool(is_causal)), int(sms),
                                          ctypes.byref(out)), "fa2_fwd_schedule_for")
    return out.value


def fa2_fwd_workspace_bytes(D: int) -> int:
    n = ctypes.c_size_t(0)
    _check(library().fa2_fwd_workspace_bytes(int(D), ctypes.byref(n)), "fa2_fwd_workspace_bytes")
    return n.value


def fa2_fwd_host_buffer_bytes(B: int, H: int, N: int, D: int) -> int:
    n = ctypes.c_size_t(0)
    _check(library().fa2_fwd_host_buffer_bytes(int(B), int(H), int(N), int(D), ctypes.byref(n)),
           "fa2_fwd_host_buffer_bytes")
    return n.value


def fa2_bwd_workspace_bytes(B: int, H: int, N: int, D: int) -> int:
    n = ctypes.c_size_t(0)
    _check(library().fa2_bwd_workspace_bytes(int(B), int(H), int(N), int(D), ctypes.byref(n)),
           "fa2_bwd_workspace_bytes")
    return n.value


def fa2_bwd(Q: int, K: int, V: int, O: int, dO: int, LSE: int, dQ: int, dK: int, dV: int, B: int, H: int, N: int,
            D: int, scale: float, is_causal: int, dtype: int, workspace: int | None, workspace_bytes: int,
            stream: int | None) -> int:
    """Pointer-level call of the backward pass; returns the raw status code."""
    return library().fa2_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, D, float(scale), int(is_causal),
                             int(dtype), workspace, int(workspace_bytes), stream)


def fa2_bwd_sched(Q: int, K: int, V: int, O: int, dO: int, LSE: int, dQ: int, dK: int, dV: int, B: int, H: int,
                  N: int, D: int, scale: float, is_causal: int, dtype: int, workspace: int | None,
                  workspace_bytes: int, schedule: int, stream: int | None) -> int:
    """Pointer-level call of the backward pass with an explicit schedule code; returns the raw status."""
    return library().fa2_bwd_sched(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, D, float(scale), int(is_causal),
                                   int(dtype), workspace, int(workspace_bytes), int(schedule), stream)


def fa2_device_status(stream: int | None = None, clear: bool = False) -> int:
    """The device watchdog word: 0, or the site id of the wait that timed out (the C call then
    returns FA2_ERR_TIMEOUT, which is reported here through the value, not raised)."""
    v = ctypes.c_int(0)
    code = library().fa2_device_status(stream, ctypes.byref(v), int(bool(clear)))
    if code != FA2_ERR_TIMEOUT:
        _check(code, "fa2_device_status")
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
_sm_counts = {}


def workspace_for(device, D: int, stream=None):
    """A cached caller-side workspace (torch uint8 tensor) for the balanced schedule on `device`.

    One per (device, head dim, stream): calls on one stream are ordered, so they
    may share it; calls on different streams get different workspaces, since
    two balanced launches that overlap on the GPU must not share one. The
    cache keeps one workspace (about 21 MB on a 152-SM GPU) per stream used.
    """
    import torch
    dev = torch.device(device)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    key = (dev.index, D, stream.cuda_stream)
    ws = _workspaces.get(key)
    if ws is None:
        with torch.cuda.device(dev):
            n = fa2_fwd_workspace_bytes(D)
        ws = torch.empty(n, dtype=torch.uint8, device=dev)
        _workspaces[key] = ws
    return ws


def sm_count(device) -> int:
    import torch
    dev = torch.device(device)
    n = _sm_counts.get(dev.index)
    if n is None:
        n = torch.cuda.get_device_properties(dev).multi_processor_count
        _sm_counts[dev.index] = n
    return n


UNIT_ROWS = 256  # query rows per work unit of the kernel (head dims up to 128)
KV_TILE = 128    # keys per K/V tile


def unit_rows(D: int = 128) -> int:
    """Query rows per work unit: 256 (two 128-row sub-tiles), or 128 at head dims from 256."""
    return KV_TILE if D >= 256 else UNIT_ROWS


def steps_per_head(N: int, is_causal: bool, D: int = 128) -> int:
    """K/V-tile steps (one work unit against one 128-key tile) of one head."""
    rows = unit_rows(D)
    sub = rows // KV_TILE
    n_qt, nkv = -(-N // rows), -(-N // KV_TILE)
    if not is_causal:
        return n_qt * nkv
    return sum(min(sub * (qt + 1), nkv) for qt in range(n_qt))


def choose_schedule(B: int, H: int, N: int, is_causal: bool, sms: int, D: int = 128) -> str:
    """The schedule the library's FA2_SCHED_AUTO takes for a problem ("units" or "balanced").

    The choice is made in C (fa2_fwd_schedule_for, the cost model of
    fa2_fwd_sched); this only names it.
    """
    code = fa2_fwd_schedule_for(B, H, N, D, is_causal, sms)
    return "balanced" if code == FA2_SCHED_BALANCED else "units"


_DTYPE_CODES = {}


def _dtype_code_of(dt) -> int:
    code = _DTYPE_CODES.get(dt)
    if code is None:
        import torch
        if dt == torch.float16:
            code = FA2_F16
        elif dt == torch.bfloat16:
            code = FA2_BF16
        else:
            raise TypeError(f"unsupported dtype {dt}; expected float16 or bfloat16")
        _DTYPE_CODES[dt] = code
    return code


def attention_forward(q, k, v, scale: float | None = None, is_causal: bool = False, out=None, lse=None,
                      stream=None, schedule: str = "auto", workspace=None):
    """FlashAttention-2 forward over torch CUDA tensors [B, H, N, D] (fp16/bf16).

    Returns (O, LSE): O like q, LSE float32 [B, H, N]. `out` / `lse` may be
    passed to write into caller-owned buffers. Runs on `stream` (a
    torch.cuda.Stream) or the current stream of q's device.
    schedule: "auto" (the library's choice, fa2_fwd_sched with FA2_SCHED_AUTO),
    "balanced" (equal work per SM, with a workspace) or "units" (whole query
    tiles per CTA in rounds, no workspace).
    workspace: optional uint8 CUDA tensor for the balanced schedule; by default
    a cached one per (device, head dim, stream) is used, so calls on different
    streams never share one.
    The checks here are the ones the C ABI cannot make (tensor metadata); the
    library checks sizes, alignment and overlap itself.
    """
    import torch
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    shape = q.shape
    if len(shape) != 4 or k.shape != shape or v.shape != shape:
        raise ValueError("q, k, v must share one [B, H, N, D] shape")
    dt = q.dtype
    if k.dtype != dt or v.dtype != dt:
        raise ValueError("q, k, v must share one dtype")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    code_sched = _SCHEDULES.get(schedule)
    if code_sched is None:
        raise ValueError("schedule must be 'auto', 'balanced' or 'units'")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k, v must be on one device")
    B, H, N, D = shape
    dtc = _dtype_code_of(dt)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != shape or out.dtype != dt or not out.is_contiguous() or out.device != q.device:
        raise ValueError("out must be a contiguous tensor like q, on its device")
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    elif lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous() or lse.device != q.device:
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor on q's device")
    dev = q.device
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    if code_sched == FA2_SCHED_UNITS:
        ws_ptr, ws_bytes = None, 0
    else:
        ws = workspace if workspace is not None else workspace_for(dev, D, s)
        ws_ptr, ws_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    lib = _lib if _lib is not None else library()
    if torch.cuda.current_device() == dev.index:
        code = lib.fa2_fwd_sched(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N,
                                 D, scale, 1 if is_causal else 0, dtc, ws_ptr, ws_bytes, code_sched, s.cuda_stream)
    else:
        with torch.cuda.device(dev):
            code = lib.fa2_fwd_sched(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H,
                                     N, D, scale, 1 if is_causal else 0, dtc, ws_ptr, ws_bytes, code_sched,
                                     s.cuda_stream)
    if code != FA2_OK:
        _check(code, "fa2_fwd_sched")
    return out, lse


HOST_CHUNKS = 16           # target number of head chunks of attention_forward_host
HOST_CHUNK_MIN_STEPS = 4096  # K/V-tile steps a chunk needs to keep the GPU busy (~27 per SM)


def host_chunk_heads(B: int, H: int, N: int, is_causal: bool, sms: int, D: int = 128) -> int:
    """Heads per chunk of the host-memory pipeline.

    The copies are the bottleneck end to end, so the pipeline wants many
    chunks (its fill and drain are one chunk's copy-in and one chunk's kernel
    and copy-out), but each chunk's kernel must still fill the GPU: at least
    HOST_CHUNK_MIN_STEPS steps, and for causal work (round schedule) at least
    one unit per SM. Measured on target-like shapes this picks the fastest of
    1-64 heads per chunk.
    """
    bh = B * H
    if bh <= 0:
        return 1
    hpc = max(-(-bh // HOST_CHUNKS), -(-HOST_CHUNK_MIN_STEPS // max(1, steps_per_head(N, is_causal, D))))
    if is_causal:
        hpc = max(hpc, -(-sms // -(-N // unit_rows(D))))
    return max(1, min(hpc, bh))


def attention_forward_host(q, k, v, scale: float | None = None, is_causal: bool = False, out=None, lse=None,
                           stream=None, device=None, heads_per_chunk: int | None = None, schedule: str = "auto",
                           device_buffer=None, synchronize: bool = True):
    """FlashAttention-2 forward over host (CPU) tensors [B, H, N, D] through fa2_fwd_host.

    The inputs are copied to `device` (default: the current CUDA device), the
    forward pass runs there and O, LSE are copied back into `out` / `lse`
    (allocated in page-locked memory when not given), chunk by chunk so that
    the copies overlap the kernels. Page-locked inputs are needed for the
    copies to overlap. Q, K, V given as the three slices of one packed
    [3, B, H, N, D] buffer take one copy per chunk instead of three, and a
    page-locked `lse` is written by the kernels in place (no copy). With synchronize=False the call returns once the work
    is enqueued on `stream`; the results are valid after that stream is
    synchronised.
    schedule: "auto" (choose_schedule applied to one chunk), "balanced" or "units".
    device_buffer: optional uint8 CUDA tensor of at least
    fa2_fwd_host_buffer_bytes(B, H, N, D) bytes; by default one is allocated.
    """
    import torch
    if q.is_cuda or k.is_cuda or v.is_cuda:
        raise ValueError("q, k, v must be host (CPU) tensors; use attention_forward for CUDA tensors")
    if q.shape != k.shape or q.shape != v.shape or q.dim() != 4:
        raise ValueError("q, k, v must share one [B, H, N, D] shape")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError("q, k, v must share one dtype")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    if schedule not in ("auto", "balanced", "units"):
        raise ValueError("schedule must be 'auto', 'balanced' or 'units'")
    B, H, N, D = q.shape
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    sms = sm_count(dev)
    hpc = host_chunk_heads(B, H, N, is_causal, sms, D) if heads_per_chunk is None else int(heads_per_chunk)
    if hpc < 1:
        raise ValueError("heads_per_chunk must be >= 1")
    if schedule == "auto":
        schedule = choose_schedule(1, min(hpc, B * H), N, is_causal, sms, D)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    if out.is_cuda or out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous host tensor like q")
    if lse.is_cuda or lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, N] host tensor")
    with torch.cuda.device(dev):
        need = fa2_fwd_host_buffer_bytes(B, H, N, D)
        buf = device_buffer if device_buffer is not None else torch.empty(need, dtype=torch.uint8, device=dev)
        if not buf.is_cuda or buf.device != dev or buf.numel() * buf.element_size() < need:
            raise ValueError(f"device_buffer must be a CUDA tensor on {dev} of at least {need} bytes")
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        code = library().fa2_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                      B, H, N, D, float(scale), int(bool(is_causal)), _dtype_code(q), hpc,
                                      int(schedule == "balanced"), buf.data_ptr(),
                                      buf.numel() * buf.element_size(), s.cuda_stream)
        _check(code, "fa2_fwd_host")
        if device_buffer is None:
            buf.record_stream(s)
        if synchronize:
            s.synchronize()
    return out, lse


def attention_backward(q, k, v, o, lse, do, scale: float | None = None, is_causal: bool = False, dq=None, dk=None,
                       dv=None, workspace=None, stream=None, schedule: str = "auto"):
    """Gradient of attention_forward w.r.t. q, k, v for an upstream gradient `do` (fa2_bwd_sched).

    q, k, v, o, do: contiguous CUDA tensors [B, H, N, D] of one dtype (fp16/bf16);
    o and lse are the forward's outputs for q, k, v (same scale and mask).
    Returns (dQ, dK, dV) like q. `dq` / `dk` / `dv` may be caller-owned
    outputs; `workspace` an optional uint8 CUDA tensor of at least
    fa2_bwd_workspace_bytes(B, H, N, D) bytes (allocated per call otherwise).
    Runs on `stream` (a torch.cuda.Stream) or the current stream.
    schedule: "auto" (the library's choice, as fa2_bwd), "units" (whole K/V
    tiles per SM in rounds) or "balanced" (equal query steps per SM).
    """
    import torch
    if schedule not in _SCHEDULES:
        raise ValueError("schedule must be 'auto', 'balanced' or 'units'")
    ts = (q, k, v, o, do)
    if not all(t.is_cuda for t in ts) or not lse.is_cuda:
        raise ValueError("q, k, v, o, do and lse must be CUDA tensors")
    if any(t.shape != q.shape for t in ts) or q.dim() != 4:
        raise ValueError("q, k, v, o, do must share one [B, H, N, D] shape")
    if any(t.dtype != q.dtype for t in ts):
        raise ValueError("q, k, v, o, do must share one dtype")
    if not all(t.is_contiguous() for t in ts):
        raise ValueError("q, k, v, o, do must be contiguous")
    B, H, N, D = q.shape
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    outs = []
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        if t is None:
            t = torch.empty_like(q)
        elif t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA tensor like q")
        outs.append(t)
    need = fa2_bwd_workspace_bytes(B, H, N, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    elif not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must be a CUDA tensor of at least {need} bytes")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        code = fa2_bwd_sched(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                             lse.data_ptr(), outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(), B, H, N,
                             D, scale, int(bool(is_causal)), _dtype_code(q), workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), _SCHEDULES[schedule], s.cuda_stream)
        _check(code, "fa2_bwd_sched")
    return tuple(outs)
