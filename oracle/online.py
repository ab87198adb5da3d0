"""The method's own tile-by-tile (m, l) recurrence, numpy fp64 — test infrastructure.

This is NOT a second oracle for the GPU path. It exists so that the tests can
check the two-pass definition in ``fa2_oracle.c`` against the recurrence the
pages state, on small inputs:

  for each block of Bc key columns (FlashAttention-2 MMA 代码学习, step 1):
    m_blk  = rowmax(S_blk)                    (S_blk = scale * Q K_blk^T, masked)
    m_new  = max(m_old, m_blk)
    P      = exp(S_blk - m_new)
    l      = exp(m_old - m_new) * l_old + rowsum(P)
    O      = exp(m_old - m_new) * O_old + P V_blk
  after the last block: O /= l, LSE = m + ln l   (CUDA book ch. 15, 15.1 and 15.3)

Masking follows the CUDA book ch. 15, 15.3: a column is masked (set to -inf
before the max) when col >= N (zero-padded tail of the last block) or, under
the causal mask, when col > row. While a row has seen only masked columns,
its running max stays -inf and the exponent base is taken as 0 instead
(section 15.3's note on the -inf guard), so exp never sees (-inf) - (-inf).
A row that never sees an allowed column ends with l = 0: O = 0, LSE = +inf.

The ``mutation`` argument deliberately plants one of the plausible mistakes
the book warns about, so a test can show the pins would catch it:
  "no_pad_mask"   padded tail columns are left unmasked (15.4.3)
  "max_init_zero" the running max starts at 0 instead of -inf (15.3 note)
  "no_rescale"    O and l are not rescaled when the max grows
"""
from __future__ import annotations

import numpy as np


def online_merge(q, k, v, scale: float, causal: bool, block: int, mutation: str | None = None):
    """q: [M, D] query rows (row ids 0..M-1), k, v: [N, D]. Returns (O [M, D], LSE [M])."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    M, D = q.shape
    N = k.shape[0]
    nblk = -(-N // block)
    pad = nblk * block - N
    kp = np.concatenate([k, np.zeros((pad, D))]) if pad else k
    vp = np.concatenate([v, np.zeros((pad, D))]) if pad else v

    m = np.full(M, 0.0 if mutation == "max_init_zero" else -np.inf)
    l = np.zeros(M)
    o = np.zeros((M, D))
    rows = np.arange(M)[:, None]
    for t in range(nblk):
        c0 = t * block
        cols = c0 + np.arange(block)[None, :]
        s = scale * (q @ kp[c0:c0 + block].T)
        masked = np.zeros_like(s, dtype=bool)
        if mutation != "no_pad_mask":
            masked |= cols >= N
        if causal:
            masked |= cols > rows
        s = np.where(masked, -np.inf, s)
        m_blk = s.max(axis=1)
        m_new = np.maximum(m, m_blk)
        base = np.where(np.isneginf(m_new), 0.0, m_new)
        p = np.exp(s - base[:, None])
        alpha = np.exp(m - base)
        if mutation == "no_rescale":
            alpha = np.ones_like(alpha)
        l = alpha * l + p.sum(axis=1)
        o = alpha[:, None] * o + p @ vp[c0:c0 + block]
        m = m_new
    out = np.zeros_like(o)
    lse = np.full(M, np.inf)
    ok = l > 0
    out[ok] = o[ok] / l[ok][:, None]
    lse[ok] = m[ok] + np.log(l[ok])
    return out, lse
