"""Pins for the gradient oracle: checks against facts fixed by the mathematics.

None of these re-types the gradient formulas. The main pin differentiates
the (separately pinned) forward oracle numerically: central differences of
the loss sum(O * dO) with respect to every input element. The others are a
library routine (torch autograd in float64 on the CPU), closed forms,
invariants of the softmax Jacobian and the causal structure. The mutation
test builds variants of the C gradient oracle with one plausible mistake
each and shows that at least one pin fails for every variant.
"""
from __future__ import annotations

import math
import os
import subprocess

import numpy as np
import pytest
import torch


def _worst(*errors) -> float:
    """The largest of the given errors, with NaN counted as the worst possible
    (the built-in max keeps its first argument when a later one is NaN)."""
    vals = [float(e) for e in errors]
    return math.inf if any(math.isnan(x) for x in vals) else max(vals)


TOL = 1e-11       # pins that hold up to fp64 rounding
FD_TOL = 1e-7     # central differences, step 1e-5 (truncation ~h^2, rounding ~eps/h)


def _rand(B, H, N, D, seed, sigma=1.0, count=4):
    g = np.random.default_rng(seed)
    return tuple(g.standard_normal((B, H, N, D)) * sigma for _ in range(count))


def _grad(oracle_mod, libpath=None):
    def f(q, k, v, do, scale, causal, **kw):
        return oracle_mod.attention_bwd(q, k, v, do, scale, causal, libpath=libpath, **kw)
    return f


# ----------------------------------------------------------------- pin battery
# Each pin takes (gradient callable, oracle module) and returns its largest
# deviation divided by its own tolerance: the real oracle keeps all below 1.

def pin_finite_differences(grad, oracle_mod):
    """dQ, dK, dV equal central differences of sum(O * dO), O from the forward oracle."""
    worst = 0.0
    h = 1e-5
    for (N, D, causal, seed, scale) in [(6, 3, False, 40, 0.7), (7, 4, True, 41, 0.5), (1, 2, False, 42, 1.0)]:
        q, k, v, do = _rand(1, 1, N, D, seed)
        r = grad(q, k, v, do, scale, causal)

        def loss(q_, k_, v_):
            O, _ = oracle_mod.attention_fwd(q_, k_, v_, scale, causal, nthreads=1)
            return float(np.sum(O * do))

        for name, idx in (("dq", 0), ("dk", 1), ("dv", 2)):
            base = [q, k, v]
            num = np.zeros((N, D))
            for i in range(N):
                for d in range(D):
                    plus = [x.copy() for x in base]
                    minus = [x.copy() for x in base]
                    plus[idx][0, 0, i, d] += h
                    minus[idx][0, 0, i, d] -= h
                    num[i, d] = (loss(*plus) - loss(*minus)) / (2 * h)
            worst = _worst(worst, np.abs(r[name][0, 0] - num).max() / FD_TOL)
    return worst


def pin_autograd(grad, oracle_mod):
    """torch autograd through softmax(scale Q K^T [+ mask]) V in float64 on the CPU."""
    worst = 0.0
    for (B, H, N, D, causal, seed) in [(1, 2, 37, 16, False, 43), (2, 1, 29, 8, True, 44),
                                       (1, 1, 64, 32, True, 45), (1, 1, 30, 96, False, 46)]:
        q, k, v, do = _rand(B, H, N, D, seed)
        scale = 1 / math.sqrt(D)
        r = grad(q, k, v, do, scale, causal)
        tq, tk, tv = (torch.from_numpy(x).requires_grad_(True) for x in (q, k, v))
        S = tq @ tk.transpose(-1, -2) * scale
        if causal:
            S = S.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
        O = torch.softmax(S, dim=-1) @ tv
        O.backward(torch.from_numpy(do))
        for name, t in (("dq", tq), ("dk", tk), ("dv", tv)):
            worst = _worst(worst, np.abs(r[name] - t.grad.numpy()).max() / TOL)
    return worst


def pin_uniform_weights(grad, oracle_mod):
    """Q = 0 or all K rows equal => uniform weights: dV_j = sum over the queries i that
    see key j of dO_i / |J(i)|; with equal K rows also dQ = 0 (dS rows sum to zero)."""
    worst = 0.0
    g = np.random.default_rng(46)
    N, D = 21, 8
    for causal in (False, True):
        for mode in ("zero_q", "same_k"):
            q = g.standard_normal((1, 1, N, D))
            k = g.standard_normal((1, 1, N, D))
            v = g.standard_normal((1, 1, N, D))
            do = g.standard_normal((1, 1, N, D))
            if mode == "zero_q":
                q[:] = 0.0
            else:
                k[:] = k[:, :, :1]
            r = grad(q, k, v, do, 0.6, causal)
            cnt = np.arange(1, N + 1) if causal else np.full(N, N)
            expect = np.zeros((N, D))
            for j in range(N):
                for i in range(j if causal else 0, N):
                    expect[j] += do[0, 0, i] / cnt[i]
            worst = _worst(worst, np.abs(r["dv"][0, 0] - expect).max() / TOL)
            if mode == "same_k":
                worst = _worst(worst, np.abs(r["dq"]).max() / TOL)
    return worst


def pin_dk_sums_to_zero(grad, oracle_mod):
    """Every row of dS sums to zero over its allowed keys, so sum_j dK_j = 0."""
    worst = 0.0
    for causal, seed in ((False, 47), (True, 48)):
        q, k, v, do = _rand(1, 2, 33, 8, seed)
        r = grad(q, k, v, do, 0.4, causal)
        scale_ref = np.abs(r["dk"]).max()
        worst = _worst(worst, np.abs(r["dk"].sum(axis=2)).max() / (TOL * max(1.0, 33 * scale_ref)))
    return worst


def pin_single_key(grad, oracle_mod):
    """N = 1: the weight is 1 whatever Q and K are, so dQ = dK = 0 and dV = dO."""
    q, k, v, do = _rand(2, 2, 1, 16, 49)
    worst = 0.0
    for causal in (False, True):
        r = grad(q, k, v, do, 0.3, causal)
        worst = _worst(worst, np.abs(r["dq"]).max() / TOL, np.abs(r["dk"]).max() / TOL,
                    np.abs(r["dv"] - do).max() / TOL)
    return worst


def pin_permutation(grad, oracle_mod):
    """Permuting K and V rows together permutes dK and dV alike and leaves dQ unchanged."""
    q, k, v, do = _rand(1, 2, 27, 8, 50)
    perm = np.random.default_rng(51).permutation(27)
    r1 = grad(q, k, v, do, 0.5, False)
    r2 = grad(q, k[:, :, perm], v[:, :, perm], do, 0.5, False)
    return _worst(np.abs(r1["dq"] - r2["dq"]).max(), np.abs(r1["dk"][:, :, perm] - r2["dk"]).max(),
               np.abs(r1["dv"][:, :, perm] - r2["dv"]).max()) / TOL


def pin_causal_structure(grad, oracle_mod):
    """Causal: dQ_i depends only on K/V rows j <= i (and Q/dO row i); dK_j and dV_j only on
    Q/dO rows i >= j. Unchanged rows keep their values bit for bit; changed ones move."""
    q, k, v, do = _rand(1, 1, 18, 8, 52)
    r1 = grad(q, k, v, do, 0.4, True)
    worst = 0.0
    for i in (0, 6, 12):
        k2, v2 = k.copy(), v.copy()
        k2[0, 0, i + 1:] += 2.0
        v2[0, 0, i + 1:] -= 1.5
        r2 = grad(q, k2, v2, do, 0.4, True)
        worst = _worst(worst, np.abs(r1["dq"][0, 0, :i + 1] - r2["dq"][0, 0, :i + 1]).max() / TOL)
        if np.abs(r1["dq"][0, 0, i + 1:] - r2["dq"][0, 0, i + 1:]).max() < 1e-6:
            worst = _worst(worst, 1e3)
        q3, do3 = q.copy(), do.copy()
        q3[0, 0, :i] += 1.0
        do3[0, 0, :i] *= -2.0
        r3 = grad(q3, k, v, do3, 0.4, True)
        worst = _worst(worst, np.abs(r1["dk"][0, 0, i:] - r3["dk"][0, 0, i:]).max() / TOL,
                    np.abs(r1["dv"][0, 0, i:] - r3["dv"][0, 0, i:]).max() / TOL)
        if i > 0 and np.abs(r1["dv"][0, 0, :i] - r3["dv"][0, 0, :i]).max() < 1e-6:
            worst = _worst(worst, 1e3)
    return worst


def pin_delta_is_dout_dot_output(grad, oracle_mod):
    """Delta_i = <dO_i, O_i> with O from the forward oracle."""
    worst = 0.0
    for causal, seed in ((False, 53), (True, 54)):
        q, k, v, do = _rand(2, 1, 25, 16, seed)
        r = grad(q, k, v, do, 0.25, causal)
        O, _ = oracle_mod.attention_fwd(q, k, v, 0.25, causal)
        worst = _worst(worst, np.abs(r["delta"] - np.einsum("bhnd,bhnd->bhn", do, O)).max() / TOL)
    return worst


def pin_magnitudes(grad, oracle_mod):
    """|x| <= x_mag for every gradient element; with dO >= 0 every term of dV is >= 0,
    so dV_mag equals dV."""
    q, k, v, do = _rand(1, 2, 30, 8, 55)
    do = np.abs(do)
    worst = 0.0
    for causal in (False, True):
        r = grad(q, k, v, do, 0.5, causal, magnitudes=True)
        for name in ("dq", "dk", "dv"):
            worst = _worst(worst, np.max(np.abs(r[name]) - r[name + "_mag"]) / TOL)
        worst = _worst(worst, np.abs(r["dv_mag"] - r["dv"]).max() / TOL)
    return worst


def pin_head_selection(grad, oracle_mod):
    """Computing a subset of heads gives exactly the full result for those heads."""
    q, k, v, do = _rand(2, 3, 17, 8, 56)
    full = grad(q, k, v, do, 0.5, True)
    part = grad(q, k, v, do, 0.5, True, heads=[5, 1])
    worst = 0.0
    for r, bh in enumerate((5, 1)):
        b, h = divmod(bh, 3)
        for name in ("dq", "dk", "dv"):
            worst = _worst(worst, np.abs(part[name][r] - full[name][b, h]).max() / TOL)
    return worst


PINS = [pin_finite_differences, pin_autograd, pin_uniform_weights, pin_dk_sums_to_zero, pin_single_key,
        pin_permutation, pin_causal_structure, pin_delta_is_dout_dot_output, pin_magnitudes,
        pin_head_selection]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(oracle_mod, pin):
    assert pin(_grad(oracle_mod), oracle_mod) < 1.0


def test_thread_count_does_not_change_results(oracle_mod):
    q, k, v, do = _rand(1, 2, 45, 16, 57)
    a = oracle_mod.attention_bwd(q, k, v, do, 0.25, True, nthreads=1)
    b = oracle_mod.attention_bwd(q, k, v, do, 0.25, True, nthreads=7)
    assert all(np.array_equal(a[n], b[n]) for n in ("dq", "dk", "dv", "delta"))


def test_gradient_oracle_rejects_bad_heads(oracle_mod):
    q, k, v, do = _rand(1, 1, 8, 4, 58)
    with pytest.raises(ValueError):
        oracle_mod.attention_bwd(q, k, v, do, 1.0, False, heads=[1])


# ----------------------------------------------- mutants of the C gradient oracle
MUTANTS = {
    "Delta dropped (dQ pass)": ("const double ds = p * (dp - delta);", "const double ds = p * dp;"),
    "Delta dropped (dK pass)": ("const double ds = p * (dp - c->delta[i]);", "const double ds = p * dp;"),
    "Delta without 1/l": ("delta += doi[col] * (o / l);", "delta += doi[col] * o;"),
    "dQ scale dropped": ("const double t = c->scale * ds * kj[col];", "const double t = ds * kj[col];"),
    "dK scale dropped": ("const double tk = c->scale * ds * qi[col];", "const double tk = ds * qi[col];"),
    "dV weighted by dS": ("const double tv = p * doi[col];", "const double tv = ds * doi[col];"),
    "dK from K": ("const double tk = c->scale * ds * qi[col];", "const double tk = c->scale * ds * kj[col];"),
    "dP from K (dK pass)": ("const double dp = dot(doi, vj, d);", "const double dp = dot(doi, kj, d);"),
    "P not normalised (dK pass)": ("exp(sij - c->m[i]) / c->l[i];", "exp(sij - c->m[i]);"),
    "causal first query off by one": ("return c->causal ? j : 0;", "return c->causal ? j + 1 : 0;"),
    "causal key count off by one": ("return (i + 1 < c->n) ? i + 1 : c->n;", "return (i + 2 < c->n) ? i + 2 : c->n;"),
    "K transposed stride (dQ pass)": ("const double *kj = c->k + j * d;\n        const double p = s[j] / l;",
                                      "const double *kj = c->k + j;\n        const double p = s[j] / l;"),
    "wrong softmax sign": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_gradient_oracle_mutants(oracle_mod, tmp_path, name):
    src_path = os.path.join(os.path.dirname(oracle_mod.__file__), "fa2_bwd_oracle.c")
    src = open(src_path).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    c_path = tmp_path / "mutant.c"
    so_path = tmp_path / "libmutant.so"
    c_path.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", str(c_path), "-o",
                    str(so_path), "-lm"], check=True)
    grad = _grad(oracle_mod, libpath=str(so_path))
    failed = []
    for pin in PINS:
        try:
            err = pin(grad, oracle_mod)
        except Exception:
            err = float("inf")
        if not (err < 1.0):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the mutant '{name}'"
