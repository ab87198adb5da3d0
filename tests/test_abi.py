"""Host-side checks of the C ABI: the library loads, exports what include/fa2.h
declares, and rejects bad arguments before touching a GPU. No kernel runs here."""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa2.h")


@pytest.fixture(scope="module")
def lib():
    from attention_forward_03_gb300 import build
    build.build()
    from attention_forward_03_gb300 import binding
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa2_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert "fa2_fwd" in names and "fa2_device_status" in names
    assert len(names) >= 6


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(so, name), f"{name} declared in fa2.h but not exported"
    assert set(declared_functions()) == set(lib.SIGNATURES), "binding signatures out of sync with fa2.h"


def test_codes_match_header(lib):
    text = open(HEADER).read()
    for name in ("FA2_F16", "FA2_BF16", "FA2_OK", "FA2_ERR_INVALID_ARG", "FA2_ERR_UNSUPPORTED",
                 "FA2_ERR_ALIGN", "FA2_ERR_CUDA", "FA2_ERR_TIMEOUT"):
        m = re.search(rf"#define {name} \(?(-?\d+)\)?", text)
        assert m and int(m.group(1)) == getattr(lib, name), name


def test_version_and_strings(lib):
    assert lib.fa2_version() >> 16 == 1
    for code in (0, -1, -2, -3, -4, -5, 17):
        assert isinstance(lib.library().fa2_error_string(code), bytes)
    assert lib.library().fa2_last_cuda_error() is not None
    lib.fa2_set_watchdog_ns(0)


A = 0x10000  # 16-byte aligned fake addresses, far apart; never dereferenced by these tests
GOOD = dict(Q=A, K=A * 16, V=A * 32, O=A * 48, LSE=A * 64, B=1, H=2, N=64, D=64, scale=0.125, is_causal=0,
            dtype=0, stream=None)


def call(lib, **over):
    a = dict(GOOD)
    a.update(over)
    return lib.fa2_fwd(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["N"], a["D"], a["scale"],
                       a["is_causal"], a["dtype"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(B=-1), -1), (dict(H=-3), -1), (dict(N=-1), -1),
    (dict(D=48), -2), (dict(D=768), -2), (dict(D=2048), -2), (dict(D=0), -2), (dict(D=16), -2), (dict(D=160), -2),
    (dict(D=192), -2), (dict(D=384), -2),
    (dict(dtype=2), -2), (dict(dtype=-1), -2),
    (dict(scale=0.0), -1), (dict(scale=-0.5), -1), (dict(scale=float("nan")), -1), (dict(scale=float("inf")), -1),
    (dict(Q=None), -1), (dict(K=None), -1), (dict(V=None), -1), (dict(O=None), -1), (dict(LSE=None), -1),
    (dict(Q=A + 8), -3), (dict(V=A * 32 + 2), -3), (dict(O=A * 48 + 4), -3), (dict(LSE=A * 64 + 12), -3),
    (dict(O=A + 64), -1),            # O overlaps Q
    (dict(LSE=A * 48 + 128), -1),    # LSE overlaps O
    (dict(B=1 << 16, H=1 << 16), -1),  # B*H overflows int32
])
def test_bad_arguments_are_rejected_before_any_gpu_work(lib, over, code):
    assert call(lib, **over) == code


def call_ws(lib, ws, ws_bytes, **over):
    a = dict(GOOD)
    a.update(over)
    return lib.fa2_fwd_ws(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["N"], a["D"], a["scale"],
                          a["is_causal"], a["dtype"], ws, ws_bytes, a["stream"])


def test_workspace_variant_checks_its_arguments(lib):
    assert call_ws(lib, A * 80 + 8, 1 << 20) == lib.FA2_ERR_ALIGN           # misaligned workspace
    assert call_ws(lib, A * 48 + 256, 1 << 20) == lib.FA2_ERR_INVALID_ARG   # workspace overlaps O
    assert call_ws(lib, A * 80, 1 << 20, D=48) == lib.FA2_ERR_UNSUPPORTED
    assert call_ws(lib, None, 0, B=0) == lib.FA2_OK
    n = ctypes.c_size_t(0)
    assert lib.library().fa2_fwd_workspace_bytes(768, ctypes.byref(n)) == lib.FA2_ERR_UNSUPPORTED
    assert lib.library().fa2_fwd_workspace_bytes(64, None) == lib.FA2_ERR_INVALID_ARG


def test_no_alloc_entry_point_checks_arguments_first(lib):
    so = lib.library()
    a = dict(GOOD)
    args = lambda **o: [dict(a, **o)[x] for x in ("Q", "K", "V", "O", "LSE", "B", "H", "N", "D", "scale",
                                                   "is_causal", "dtype", "stream")]  # noqa: E731
    assert so.fa2_fwd_noalloc(*args(B=-1)) == lib.FA2_ERR_INVALID_ARG
    assert so.fa2_fwd_noalloc(*args(D=80)) == lib.FA2_ERR_UNSUPPORTED
    assert so.fa2_fwd_noalloc(*args(dtype=5)) == lib.FA2_ERR_UNSUPPORTED
    assert so.fa2_fwd_noalloc(*args(N=0)) == lib.FA2_OK


def test_host_entry_point_checks_arguments_first(lib):
    so = lib.library()
    H1, H2, H3, H4, H5 = (A * i for i in (100, 116, 132, 148, 164))  # fake host addresses, never touched
    base = dict(Q=H1, K=H2, V=H3, O=H4, LSE=H5, B=1, H=2, N=64, D=64, scale=0.125, is_causal=0, dtype=0, hpc=0,
                balanced=0, buf=A * 256, nbuf=1 << 30, stream=None)

    def host(**o):
        a = dict(base, **o)
        return so.fa2_fwd_host(*[a[x] for x in ("Q", "K", "V", "O", "LSE", "B", "H", "N", "D", "scale", "is_causal",
                                                "dtype", "hpc", "balanced", "buf", "nbuf", "stream")])
    assert host(B=-1) == lib.FA2_ERR_INVALID_ARG
    assert host(hpc=-2) == lib.FA2_ERR_INVALID_ARG
    assert host(D=48) == lib.FA2_ERR_UNSUPPORTED
    assert host(dtype=3) == lib.FA2_ERR_UNSUPPORTED
    assert host(scale=0.0) == lib.FA2_ERR_INVALID_ARG
    assert host(Q=None) == lib.FA2_ERR_INVALID_ARG
    assert host(buf=None) == lib.FA2_ERR_INVALID_ARG
    assert host(buf=A * 256 + 128) == lib.FA2_ERR_ALIGN
    assert host(O=H1 + 64) == lib.FA2_ERR_INVALID_ARG      # O overlaps Q
    assert host(LSE=H4 + 16) == lib.FA2_ERR_INVALID_ARG    # LSE overlaps O
    assert host(B=0) == lib.FA2_OK and host(N=0, Q=None, buf=None) == lib.FA2_OK
    n = ctypes.c_size_t(0)
    assert so.fa2_fwd_host_buffer_bytes(1, 2, 64, 64, None) == lib.FA2_ERR_INVALID_ARG
    assert so.fa2_fwd_host_buffer_bytes(1, 2, 64, 768, ctypes.byref(n)) == lib.FA2_ERR_UNSUPPORTED
    assert so.fa2_fwd_host_buffer_bytes(-1, 2, 64, 64, ctypes.byref(n)) == lib.FA2_ERR_INVALID_ARG


def test_host_chunking_rule():
    from attention_forward_03_gb300.binding import HOST_CHUNKS, host_chunk_heads, steps_per_head
    # one K/V tile per 128 keys, one unit per 256 queries; causal unit qt sees 2qt+2 tiles
    assert steps_per_head(8192, False) == 32 * 64
    assert steps_per_head(512, True) == 2 + 4 and steps_per_head(300, True) == 2 + 3
    assert steps_per_head(8192, False, 256) == 64 * 64
    assert steps_per_head(512, True, 256) == 1 + 2 + 3 + 4 and steps_per_head(300, True, 256) == 1 + 2 + 3
    assert host_chunk_heads(1, 1, 128, False, 152) == 1
    # the shapes the host pipeline was measured on, and the fastest chunking found
    assert host_chunk_heads(1, 8, 8192, False, 152) == 2
    assert host_chunk_heads(4, 16, 8192, False, 152) == 4
    assert host_chunk_heads(1, 4, 32768, True, 152) == 2
    assert host_chunk_heads(4, 16, 4096, True, 152) == 16
    for B, H, N, c in ((1, 8, 8192, False), (4, 16, 8192, False), (2, 12, 1000, False), (1, 4, 300, True),
                       (3, 7, 64, False)):
        hpc = host_chunk_heads(B, H, N, c, 152)
        assert 1 <= hpc <= B * H and -(-(B * H) // hpc) <= HOST_CHUNKS


@pytest.mark.parametrize("over", [dict(B=0), dict(H=0), dict(N=0),
                                  dict(B=0, Q=None, K=None, V=None, O=None, LSE=None)])
def test_empty_problem_is_a_no_op(lib, over):
    assert call(lib, **over) == lib.FA2_OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful on a host without a GPU")
def test_valid_call_without_a_gpu_fails_loudly(lib):
    assert call(lib) == lib.FA2_ERR_CUDA
    # every supported head dimension passes the argument checks and reaches the device query
    for d in (32, 64, 96, 128, 256, 512, 1024):
        assert call(lib, D=d) == lib.FA2_ERR_CUDA
        assert call_ws(lib, A * 80, 1 << 24, D=d) == lib.FA2_ERR_CUDA
    assert lib.library().fa2_last_cuda_error().decode() != ""
    with pytest.raises(lib.Fa2Error):
        lib._check(call(lib), "fa2_fwd")


def test_binding_refuses_cpu_tensors(lib):
    q = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        lib.attention_forward(q, q, q)


def test_missing_library_raises(lib, monkeypatch, tmp_path):
    import attention_forward_03_gb300.binding as b
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        b.library()


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "attention_forward_03_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f
                assert "fa2_oracle" not in text, f


def test_schedule_choice(lib):
    # the binding names the choice the C cost model (fa2_fwd_schedule_for) makes
    from attention_forward_03_gb300.binding import choose_schedule
    assert choose_schedule(1, 8, 8192, False, 152) == "balanced"   # 256 units: 2 rounds of 64 vs 112 steps
    assert choose_schedule(4, 16, 8192, False, 152) == "units"     # 2048 units: 14 rounds of 64 vs 866 steps
    assert choose_schedule(1, 8, 8192, True, 152) == "units"       # causal: zig-zag rounds
    assert choose_schedule(2, 12, 1000, False, 152) == "units"     # 8-tile units: 8 vs 9 steps
    assert choose_schedule(1, 152, 256, False, 152) == "units"     # exactly one full round
    assert choose_schedule(1, 1, 8192, False, 152) == "balanced"   # 32 long units on 152 SMs
    assert choose_schedule(1, 1, 128, False, 152) == "units"       # one tiny unit
    assert choose_schedule(0, 8, 8192, False, 152) == "units"      # empty
    # head dim 256: 128-row units (one sub-tile)
    assert choose_schedule(1, 8, 8192, False, 152, 256) == "balanced"  # 512 units: 4 rounds of 64 vs 220 steps
    assert choose_schedule(1, 19, 1024, False, 152, 256) == "units"    # exactly one full round
    # head dims 512 and 1024 run on the round schedule only
    assert choose_schedule(1, 8, 8192, False, 152, 512) == "units"
    assert choose_schedule(1, 1, 8192, False, 152, 1024) == "units"


def test_schedule_for_arguments(lib):
    so = lib.library()
    out = ctypes.c_int(-7)
    assert so.fa2_fwd_schedule_for(1, 8, 8192, 128, 0, 152, None) == lib.FA2_ERR_INVALID_ARG
    for bad in (dict(B=-1), dict(H=-1), dict(N=-1), dict(sms=0)):
        a = dict(B=1, H=8, N=8192, sms=152, **{})
        a.update(bad)
        assert so.fa2_fwd_schedule_for(a["B"], a["H"], a["N"], 128, 0, a["sms"], ctypes.byref(out)) == -1
    assert so.fa2_fwd_schedule_for(1, 8, 8192, 48, 0, 152, ctypes.byref(out)) == lib.FA2_ERR_UNSUPPORTED
    assert out.value == -7  # untouched on error
    assert so.fa2_fwd_schedule_for(1, 8, 8192, 128, 0, 152, ctypes.byref(out)) == lib.FA2_OK
    assert out.value == lib.FA2_SCHED_BALANCED
    # the cost model at the SM-count boundary: 152 units of 8 tiles fill one round exactly
    assert lib.fa2_fwd_schedule_for(1, 38, 1024, 128, False, 152) == lib.FA2_SCHED_UNITS
    assert lib.fa2_fwd_schedule_for(1, 39, 1024, 128, False, 152) == lib.FA2_SCHED_BALANCED


def call_sched(lib, schedule, ws=None, nws=0, **over):
    a = dict(GOOD)
    a.update(over)
    return lib.library().fa2_fwd_sched(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["N"], a["D"],
                                       a["scale"], a["is_causal"], a["dtype"], ws, nws, schedule, a["stream"])


def test_forward_schedule_codes(lib):
    for bad in (-1, 3, 9):
        assert call_sched(lib, bad) == lib.FA2_ERR_INVALID_ARG
    # the balanced schedule needs a workspace (the rounds and auto do not)
    assert call_sched(lib, lib.FA2_SCHED_BALANCED) == lib.FA2_ERR_INVALID_ARG
    assert call_sched(lib, lib.FA2_SCHED_BALANCED, B=0) == lib.FA2_OK
    # the usual argument checks come before any device work
    assert call_sched(lib, lib.FA2_SCHED_AUTO, D=48) == lib.FA2_ERR_UNSUPPORTED
    assert call_sched(lib, lib.FA2_SCHED_UNITS, Q=A + 8) == lib.FA2_ERR_ALIGN
    assert call_sched(lib, lib.FA2_SCHED_AUTO, A * 80, 1 << 24, scale=0.0) == lib.FA2_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful on a host without a GPU")
def test_schedule_calls_and_status_without_a_gpu_fail_loudly(lib):
    for sched in (lib.FA2_SCHED_AUTO, lib.FA2_SCHED_UNITS):
        assert call_sched(lib, sched) == lib.FA2_ERR_CUDA
    assert call_sched(lib, lib.FA2_SCHED_AUTO, A * 80, 1 << 24) == lib.FA2_ERR_CUDA
    assert call_sched(lib, lib.FA2_SCHED_BALANCED, A * 80, 1 << 24) == lib.FA2_ERR_CUDA
    v = ctypes.c_int(0)
    assert lib.library().fa2_device_status(None, ctypes.byref(v), 0) == lib.FA2_ERR_CUDA


BWD = dict(Q=A, K=A * 16, V=A * 32, O=A * 48, dO=A * 64, LSE=A * 80, dQ=A * 96, dK=A * 112, dV=A * 128, B=1, H=2,
           N=64, D=64, scale=0.125, is_causal=0, dtype=0, ws=A * 144, nws=1 << 24, stream=None)


def call_bwd(lib, **over):
    a = dict(BWD, **over)
    return lib.library().fa2_bwd(*[a[x] for x in ("Q", "K", "V", "O", "dO", "LSE", "dQ", "dK", "dV", "B", "H", "N",
                                                  "D", "scale", "is_causal", "dtype", "ws", "nws", "stream")])


@pytest.mark.parametrize("over,code", [
    (dict(B=-1), -1), (dict(N=-2), -1), (dict(D=48), -2), (dict(D=256), -2), (dict(dtype=7), -2),
    (dict(scale=0.0), -1), (dict(scale=float("nan")), -1),
    (dict(Q=None), -1), (dict(dO=None), -1), (dict(LSE=None), -1), (dict(dK=None), -1), (dict(ws=None), -1),
    (dict(dO=A * 64 + 8), -3), (dict(dV=A * 128 + 4), -3), (dict(ws=A * 144 + 16), -3),
    (dict(nws=1024), -1),                 # workspace too small
    (dict(dQ=A + 512), -1),               # dQ overlaps Q
    (dict(dK=A * 96 + 256), -1),          # dK overlaps dQ
    (dict(ws=A * 128 + 256), -1),         # workspace overlaps dV
    (dict(B=1 << 16, H=1 << 16), -1),     # B*H overflows int32
])
def test_backward_rejects_bad_arguments_before_any_gpu_work(lib, over, code):
    assert call_bwd(lib, **over) == code


def test_backward_empty_problem_and_workspace_size(lib):
    assert call_bwd(lib, B=0) == lib.FA2_OK
    assert call_bwd(lib, N=0, Q=None, ws=None) == lib.FA2_OK
    # fp32 dQ accumulator [B,H,N,D] + LSE*log2(e) and Delta rows padded to the step height (128 rows at
    # head dims up to 64, else 64) + the balanced schedule's 160 partial slots of 2*128*D floats and their
    # 160 flags, each rounded to 256 bytes
    r256 = lambda x: -(-x // 256) * 256  # noqa: E731
    for (B, H, N, D) in ((1, 2, 64, 64), (2, 12, 1000, 64), (1, 8, 8192, 128), (1, 1, 1, 128), (1, 3, 200, 96)):
        sr = 128 if D <= 64 else 64
        npad = -(-N // sr) * sr
        assert lib.fa2_bwd_workspace_bytes(B, H, N, D) == (r256(B * H * N * D * 4) + 2 * r256(B * H * npad * 4)
                                                           + r256(160 * 2 * 128 * D * 4) + r256(160 * 8))
    n = ctypes.c_size_t(0)
    assert lib.library().fa2_bwd_workspace_bytes(1, 1, 64, 256, ctypes.byref(n)) == lib.FA2_ERR_UNSUPPORTED
    for D in (32, 96):  # the padded head dims
        npad = 128 if D <= 64 else 64
        assert lib.fa2_bwd_workspace_bytes(1, 1, 64, D) == (r256(64 * D * 4) + 2 * r256(npad * 4)
                                                            + r256(160 * 2 * 128 * D * 4) + r256(160 * 8))
    assert lib.library().fa2_bwd_workspace_bytes(1, 1, 64, 64, None) == lib.FA2_ERR_INVALID_ARG


def test_backward_schedule_codes(lib):
    a = dict(BWD)
    args = [a[x] for x in ("Q", "K", "V", "O", "dO", "LSE", "dQ", "dK", "dV", "B", "H", "N", "D", "scale",
                           "is_causal", "dtype", "ws", "nws")]
    so = lib.library()
    for bad in (-1, 3, 7):
        assert so.fa2_bwd_sched(*args, bad, None) == lib.FA2_ERR_INVALID_ARG
    assert so.fa2_bwd_sched(*args[:9], 0, *args[10:], lib.FA2_SCHED_BALANCED, None) == lib.FA2_OK  # B = 0
    assert (lib.FA2_SCHED_AUTO, lib.FA2_SCHED_UNITS, lib.FA2_SCHED_BALANCED) == (0, 1, 2)
    q = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        lib.attention_backward(q, q, q, q, torch.zeros(1, 1, 8), q, schedule="fastest")


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful on a host without a GPU")
def test_backward_without_a_gpu_fails_loudly(lib):
    assert call_bwd(lib) == lib.FA2_ERR_CUDA
