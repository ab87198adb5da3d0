"""ctypes wrapper over the gradient oracle (``fa2_bwd_oracle.c``) — test infrastructure.

The gradient of the forward definition (fp64, from the exact 16-bit values),
for an upstream gradient dO of the output:
  P = softmax(scale * Q K^T) over the allowed keys, O = P V
  dV = P^T dO,  dP = dO V^T,  Delta_i = <dO_i, O_i>,  dS = P * (dP - Delta)
  dQ = scale * dS K,  dK = scale * dS^T Q
Sources: the yangyitao.com CUDA book, ch. 15 (section 15.1, change 4: the
backward keeps LSE and recomputes S and P; the chapter's closing paragraph:
dQ accumulated across key tiles, outer loop over K/V).
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build
from .reference import _f64, default_threads

_libs = {}


def _load(path: str | None = None):
    path = path or _build.build_bwd()
    lib = _libs.get(path)
    if lib is None:
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.fa2_oracle_bwd_head.argtypes = [dp, dp, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_double,
                                            ctypes.c_int, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
        lib.fa2_oracle_bwd_head.restype = ctypes.c_int
        _libs[path] = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def attention_bwd(q, k, v, do, scale: float, causal: bool, heads=None, magnitudes: bool = False,
                  nthreads: int | None = None, libpath: str | None = None):
    """Oracle gradient of the forward pass.

    q, k, v, do: [B, H, N, D] tensors or arrays (any float dtype; widened exactly).
    heads: None for every head, else a list of flat head ids bh = b*H + h.
    magnitudes: also return per-element condition sums (dq_mag, dk_mag, dv_mag):
      a relative perturbation u of every P, dS and O value moves an element by
      at most about u times its sum (see fa2_bwd_oracle.c); each is at least
      the sum of the absolute values of the element's terms.
    libpath: load the C code from another build of it (mutation tests only).
    Returns a dict of float64 arrays: dq, dk, dv ([B,H,N,D], or [len(heads),N,D]),
    delta ([B,H,N] or [len(heads),N]) and, with magnitudes, dq_mag, dk_mag, dv_mag.
    """
    lib = _load(libpath)
    nthreads = nthreads or default_threads()
    shape = tuple(q.shape)
    B, H, N, D = shape
    ids = list(range(B * H)) if heads is None else [int(x) for x in heads]
    if any(x < 0 or x >= B * H for x in ids):
        raise ValueError("head id outside [0, B*H)")
    names = ["dq", "dk", "dv"] + (["dq_mag", "dk_mag", "dv_mag"] if magnitudes else [])
    out = {n: np.zeros((len(ids), N, D), dtype=np.float64) for n in names}
    out["delta"] = np.zeros((len(ids), N), dtype=np.float64)
    for r, bh in enumerate(ids):
        b, h = divmod(bh, H)
        qh, kh, vh, dh = (_f64(t[b, h]) for t in (q, k, v, do))
        mags = [out[n][r] for n in ("dq_mag", "dk_mag", "dv_mag")] if magnitudes else [None] * 3
        rc = lib.fa2_oracle_bwd_head(_ptr(qh), _ptr(kh), _ptr(vh), _ptr(dh), N, D, float(scale),
                                     int(bool(causal)), _ptr(out["dq"][r]), _ptr(out["dk"][r]),
                                     _ptr(out["dv"][r]), _ptr(out["delta"][r]), *(_ptr(m) for m in mags),
                                     int(nthreads))
        if rc != 0:
            raise ValueError("gradient oracle rejected its arguments")
    if heads is None:
        for n in list(out):
            out[n] = out[n].reshape((B, H) + out[n].shape[1:])
    return out


def loss_for_gradient(o, do) -> float:
    """The scalar loss whose gradient the oracle returns: sum(O * dO) (fp64)."""
    return float(np.sum(np.asarray(o, dtype=np.float64) * np.asarray(do, dtype=np.float64)))


__all__ = ["attention_bwd", "loss_for_gradient"]

