"""ctypes wrapper over the C oracle (``fa2_oracle.c``) — test infrastructure.

The definition it computes (fp64, from the exact 16-bit input values):
  s_j = scale * <Q_i, K_j>  over the allowed keys J(i) (j < N; j <= i if causal)
  O_i = sum_j exp(s_j - m) V_j / l,  LSE_i = m + ln l,  m = max s_j, l = sum exp(s_j - m)
Sources: "FlashAttention-2 MMA 代码学习", steps 0-1; yangyitao.com CUDA book
ch. 15, sections 15.1 (LSE) and 15.3 (scale, causal and column masks, the
all-masked row).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import build as _build

_libs = {}


def _load(path: str | None = None):
    """Load the oracle library (or, for the mutation tests, a variant built elsewhere)."""
    path = path or _build.build()
    lib = _libs.get(path)
    if lib is None:
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lp = ctypes.POINTER(ctypes.c_long)
        lib.fa2_oracle_head.argtypes = [dp, dp, dp, ctypes.c_long, ctypes.c_long,
                                        ctypes.c_double, ctypes.c_int, lp, ctypes.c_long,
                                        dp, dp, ctypes.c_int]
        lib.fa2_oracle_head.restype = ctypes.c_int
        _libs[path] = lib
    return lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _f64(t) -> np.ndarray:
    """Exact widening of a 16-bit (or wider) tensor/array to a contiguous float64 array."""
    if isinstance(t, torch.Tensor):
        return np.ascontiguousarray(t.detach().to("cpu", torch.float64).numpy())
    return np.ascontiguousarray(np.asarray(t, dtype=np.float64))


def _head(qh, kh, vh, scale, causal, rows, nthreads, libpath=None):
    lib = _load(libpath)
    n, d = kh.shape
    dp = ctypes.POINTER(ctypes.c_double)
    if rows is None:
        nrows = n
        rows_arr = None
        rows_ptr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.shape[0]
        rows_ptr = rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_long))
    o = np.zeros((nrows, d), dtype=np.float64)
    lse = np.zeros((nrows,), dtype=np.float64)
    rc = lib.fa2_oracle_head(qh.ctypes.data_as(dp), kh.ctypes.data_as(dp), vh.ctypes.data_as(dp),
                             n, d, float(scale), int(bool(causal)), rows_ptr, nrows,
                             o.ctypes.data_as(dp), lse.ctypes.data_as(dp), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return o, lse


def attention_fwd(q, k, v, scale: float, causal: bool, rows=None, nthreads: int | None = None,
                  libpath: str | None = None):
    """Oracle forward pass.

    q, k, v: [B, H, N, D] tensors or arrays (any float dtype; widened exactly).
    rows: None for every row, else an int array of flat row ids r = (b*H + h)*N + i.
    libpath: load the C code from another build of it (mutation tests only).
    Returns (O, LSE) as float64 numpy arrays: [B, H, N, D] and [B, H, N] when rows
    is None, else [len(rows), D] and [len(rows)] in the order given.
    """
    nthreads = nthreads or default_threads()
    if isinstance(q, torch.Tensor):
        B, H, N, D = q.shape
    else:
        B, H, N, D = np.asarray(q).shape
    if rows is None:
        O = np.zeros((B, H, N, D), dtype=np.float64)
        L = np.zeros((B, H, N), dtype=np.float64)
        for b in range(B):
            for h in range(H):
                o, l = _head(_f64(q[b, h]), _f64(k[b, h]), _f64(v[b, h]), scale, causal, None, nthreads,
                             libpath)
                O[b, h] = o
                L[b, h] = l
        return O, L
    rows = np.asarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= B * H * N):
        raise ValueError("row id outside [0, B*H*N)")
    O = np.zeros((rows.shape[0], D), dtype=np.float64)
    L = np.zeros((rows.shape[0],), dtype=np.float64)
    heads = rows // N
    for bh in np.unique(heads):
        sel = np.nonzero(heads == bh)[0]
        b, h = divmod(int(bh), H)
        o, l = _head(_f64(q[b, h]), _f64(k[b, h]), _f64(v[b, h]), scale, causal,
                     rows[sel] - bh * N, nthreads, libpath)
        O[sel] = o
        L[sel] = l
    return O, L


def sample_rows(B: int, H: int, N: int, count: int, seed: int = 0, tile: int = 128) -> np.ndarray:
    """Flat row ids for sampled parity checks at full size.

    Always includes the first and last row of the first and last head and
    rows on both sides of every tile boundary of one head, plus ``count``
    uniformly drawn rows.
    """
    rng = np.random.default_rng(seed)
    total = B * H * N
    picks = set(int(x) for x in rng.integers(0, total, size=count))
    for bh in (0, B * H - 1):
        for i in (0, 1, N - 2, N - 1):
            if 0 <= i < N:
                picks.add(bh * N + i)
    bh = int(rng.integers(0, B * H))
    for t in range(tile, N, tile * max(1, (N // tile) // 8)):
        for i in (t - 1, t):
            picks.add(bh * N + i)
    return np.array(sorted(picks), dtype=np.int64)
