"""Pins for the CPU oracle: checks against facts the pages and mathematics fix.

None of these re-types the oracle's formula. Each pin is a closed form, an
invariant, brute force on tiny inputs, the method's own tile recurrence, or a
library routine that reduces to the same definition. The mutation test at the
end builds variants of the C oracle with one plausible mistake each and shows
that at least one pin fails for every variant.
"""
from __future__ import annotations

import json
import math
import os
import re
import subprocess

import numpy as np
import pytest
import torch

import workloads


def _worst(*errors) -> float:
    """The largest of the given errors, with NaN counted as the worst possible
    (the built-in max keeps its first argument when a later one is NaN)."""
    vals = [float(e) for e in errors]
    return math.inf if any(math.isnan(x) for x in vals) else max(vals)


GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = 1e-11


def _attn(oracle_mod, libpath=None):
    def f(q, k, v, scale, causal, rows=None):
        return oracle_mod.attention_fwd(q, k, v, scale, causal, rows=rows, libpath=libpath)
    return f


def _rand(B, H, N, D, seed, sigma=1.0):
    g = np.random.default_rng(seed)
    return tuple(g.standard_normal((B, H, N, D)) * sigma for _ in range(3))


# ----------------------------------------------------------------- pin battery
# Each pin takes an attention callable and returns the largest deviation from
# what the pin fixes. The real oracle must keep every one below TOL.

def pin_closed_forms(attn):
    worst = 0.0
    with open(os.path.join(GOLDEN, "closed_forms.json")) as fh:
        cases = json.load(fh)["cases"]
    ev = lambda e: eval(e, {"math": math})  # noqa: E731  (expressions from the fixture)
    for c in cases:
        Q = np.array([[ev(x) for x in r] for r in c["Q"]], dtype=np.float64)
        K = np.array([[ev(x) for x in r] for r in c["K"]], dtype=np.float64)
        V = np.array([[ev(x) for x in r] for r in c["V"]], dtype=np.float64)
        n = K.shape[0]
        m = Q.shape[0]
        if m < n:  # query rows are the first rows of a longer sequence
            Q = np.concatenate([Q, np.zeros((n - m, Q.shape[1]))])
        O, L = attn(Q[None, None], K[None, None], V[None, None], c["scale"], c["causal"])
        Oexp = np.array([[ev(x) for x in r] for r in c["O"]])
        Lexp = np.array([ev(x) for x in c["LSE"]])
        worst = _worst(worst, np.abs(O[0, 0, :m] - Oexp).max(), np.abs(L[0, 0, :m] - Lexp).max())
    return worst


def pin_online_merge(attn, oracle_mod):
    worst = 0.0
    for (N, D, causal, block, seed, sigma) in [(37, 8, False, 8, 1, 1.0), (64, 16, True, 16, 2, 1.0),
                                               (50, 4, True, 7, 3, 3.0), (33, 8, False, 32, 4, 2.0),
                                               (1, 8, False, 4, 5, 1.0), (96, 8, True, 32, 6, 1.0)]:
        q, k, v = _rand(1, 1, N, D, seed, sigma)
        scale = 1 / math.sqrt(D)
        O, L = attn(q, k, v, scale, causal)
        o2, l2 = oracle_mod.online_merge(q[0, 0], k[0, 0], v[0, 0], scale, causal, block)
        worst = _worst(worst, np.abs(O[0, 0] - o2).max(), np.abs(L[0, 0] - l2).max())
    # every score far below zero (the running-max initialisation case); LSE is ~ -1e3
    # there, so its agreement is checked relative to its size
    q, k, v = _rand(1, 1, 40, 8, 7)
    q, k = np.abs(q), -np.abs(k) * 1e3
    O, L = attn(q, k, v, 1.0, False)
    o2, l2 = oracle_mod.online_merge(q[0, 0], k[0, 0], v[0, 0], 1.0, False, 8)
    rel = np.abs(L[0, 0] - l2).max() / max(1.0, np.abs(l2).max())
    worst = _worst(worst, np.abs(O[0, 0] - o2).max(), rel)
    return worst


def pin_identical_keys(attn):
    """All K rows equal => uniform weights: O_i = mean of the allowed V rows, LSE_i = s + ln|J(i)|."""
    worst = 0.0
    for causal in (False, True):
        g = np.random.default_rng(11)
        N, D = 23, 8
        q = g.standard_normal((1, 1, N, D))
        k = np.tile(g.standard_normal((1, 1, 1, D)), (1, 1, N, 1))
        v = g.standard_normal((1, 1, N, D))
        scale = 0.3
        O, L = attn(q, k, v, scale, causal)
        for i in range(N):
            cnt = i + 1 if causal else N
            s = scale * float(q[0, 0, i] @ k[0, 0, 0])
            worst = _worst(worst, np.abs(O[0, 0, i] - v[0, 0, :cnt].mean(axis=0)).max(),
                        abs(L[0, 0, i] - (s + math.log(cnt))))
    return worst


def pin_zero_query(attn):
    """Q = 0 => O = mean(V), LSE = ln N (non-causal)."""
    g = np.random.default_rng(12)
    N, D = 19, 16
    q = np.zeros((1, 2, N, D))
    k = g.standard_normal((1, 2, N, D))
    v = g.standard_normal((1, 2, N, D))
    O, L = attn(q, k, v, 0.25, False)
    return _worst(np.abs(O - v.mean(axis=2, keepdims=True)).max(), np.abs(L - math.log(N)).max())


def pin_permutation(attn):
    """Permuting K and V rows together leaves O and LSE unchanged (non-causal)."""
    q, k, v = _rand(2, 2, 31, 8, 13)
    perm = np.random.default_rng(14).permutation(31)
    O1, L1 = attn(q, k, v, 0.5, False)
    O2, L2 = attn(q, k[:, :, perm], v[:, :, perm], 0.5, False)
    return _worst(np.abs(O1 - O2).max(), np.abs(L1 - L2).max())


def pin_causal_prefix(attn):
    """Under the causal mask, row i depends only on K/V rows j <= i; rows keep their values
    (bit for bit) when later K/V rows change, and do change when an earlier row changes."""
    q, k, v = _rand(1, 1, 20, 8, 15)
    O1, L1 = attn(q, k, v, 0.4, True)
    worst = 0.0
    for i in (0, 5, 13):
        k2, v2 = k.copy(), v.copy()
        k2[0, 0, i + 1:] += 3.0
        v2[0, 0, i + 1:] -= 2.0
        O2, L2 = attn(q, k2, v2, 0.4, True)
        worst = _worst(worst, np.abs(O1[0, 0, :i + 1] - O2[0, 0, :i + 1]).max(),
                    np.abs(L1[0, 0, :i + 1] - L2[0, 0, :i + 1]).max())
        # the changed rows must move (a mask that hid everything would pass the line above)
        if np.abs(O1[0, 0, i + 1:] - O2[0, 0, i + 1:]).max() < 1e-6:
            worst = _worst(worst, 1.0)
    return worst


def pin_dominant_logit(attn):
    """One logit far above the rest: O is that V row within e^-gap * (N-1) * 2*max|V|."""
    g = np.random.default_rng(16)
    N, D = 17, 8
    q = g.standard_normal((1, 1, N, D))
    k = g.standard_normal((1, 1, N, D)) * 0.1
    v = g.standard_normal((1, 1, N, D))
    i, j = 3, 11
    k[0, 0, j] = q[0, 0, i] * 40.0
    O, L = attn(q, k, v, 1.0, False)
    s = q[0, 0, i] @ k[0, 0].T
    gap = s[j] - np.max(np.delete(s, j))
    bound = math.exp(-gap) * (N - 1) * 2 * np.abs(v).max()
    err = np.abs(O[0, 0, i] - v[0, 0, j]).max()
    lse_err = abs(L[0, 0, i] - s[j])  # LSE -> max logit, error <= ln(1 + (N-1) e^-gap)
    return _worst(0.0, err - bound, lse_err - math.log1p((N - 1) * math.exp(-gap)))


def pin_single_key(attn):
    """N = 1: O = V, LSE = scale * <Q0, K0>."""
    q, k, v = _rand(2, 3, 1, 16, 17)
    O, L = attn(q, k, v, 0.7, False)
    s = 0.7 * np.einsum("bhnd,bhnd->bhn", q, k)
    Oc, Lc = attn(q, k, v, 0.7, True)
    return _worst(np.abs(O - v).max(), np.abs(L - s).max(), np.abs(Oc - v).max(), np.abs(Lc - s).max())


def pin_library_softmax(attn):
    """torch.softmax / logsumexp in float64 on the CPU (a textbook routine) on small shapes."""
    worst = 0.0
    for (B, H, N, D, causal, seed) in [(1, 2, 45, 16, False, 18), (2, 1, 33, 8, True, 19),
                                       (1, 1, 128, 64, False, 20), (1, 1, 70, 32, True, 21),
                                       (1, 1, 40, 96, True, 23), (1, 2, 36, 256, False, 24)]:
        q, k, v = _rand(B, H, N, D, seed)
        scale = 1 / math.sqrt(D)
        O, L = attn(q, k, v, scale, causal)
        S = torch.from_numpy(q) @ torch.from_numpy(k).transpose(-1, -2) * scale
        if causal:
            S = S.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
        P = torch.softmax(S, dim=-1)
        Oref = (P @ torch.from_numpy(v)).numpy()
        Lref = torch.logsumexp(S, dim=-1).numpy()
        worst = _worst(worst, np.abs(O - Oref).max(), np.abs(L - Lref).max())
    return worst


def pin_row_sampling(attn):
    """Computing a sample of rows gives exactly the full result at those rows."""
    q, k, v = _rand(2, 3, 41, 8, 22)
    O, L = attn(q, k, v, 0.5, True)
    rows = np.array([0, 40, 41, 100, 245, 200, 77])
    Os, Ls = attn(q, k, v, 0.5, True, rows=rows)
    Of = O.reshape(-1, 8)[rows]
    Lf = L.reshape(-1)[rows]
    return _worst(np.abs(Os - Of).max(), np.abs(Ls - Lf).max())


PINS = [pin_closed_forms, pin_identical_keys, pin_zero_query, pin_permutation, pin_causal_prefix,
        pin_dominant_logit, pin_single_key, pin_library_softmax, pin_row_sampling]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(oracle_mod, pin):
    assert pin(_attn(oracle_mod)) < TOL


def test_pin_online_merge(oracle_mod):
    assert pin_online_merge(_attn(oracle_mod), oracle_mod) < TOL


def test_thread_count_does_not_change_results(oracle_mod):
    q, k, v = _rand(1, 2, 77, 16, 23)
    O1, L1 = oracle_mod.attention_fwd(q, k, v, 0.25, True, nthreads=1)
    O8, L8 = oracle_mod.attention_fwd(q, k, v, 0.25, True, nthreads=8)
    assert np.array_equal(O1, O8) and np.array_equal(L1, L8)


def test_sixteen_bit_inputs_are_widened_exactly(oracle_mod):
    w = workloads.custom(1, 1, 64, 64, "bf16", seed=3)
    q, k, v = workloads.make_inputs(w)
    O1, L1 = oracle_mod.attention_fwd(q, k, v, w.scale, False)
    O2, L2 = oracle_mod.attention_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), w.scale, False)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_oracle_rejects_bad_rows(oracle_mod):
    q, k, v = _rand(1, 1, 8, 4, 1)
    with pytest.raises(ValueError):
        oracle_mod.attention_fwd(q, k, v, 1.0, False, rows=np.array([8]))


# ------------------------------------------------------ the recurrence's traps
@pytest.mark.parametrize("mutation,case", [("no_pad_mask", "ragged"), ("max_init_zero", "negative"),
                                           ("no_rescale", "random")])
def test_online_merge_mutations_are_caught(oracle_mod, mutation, case):
    """The traps the CUDA book names (unmasked padded columns, a running max initialised to 0,
    a missing rescale) each change the recurrence's result against the definition."""
    if case == "ragged":
        q, k, v = _rand(1, 1, 37, 8, 30)
        scale, block = 0.35, 16
    elif case == "negative":
        q, k, v = _rand(1, 1, 40, 8, 31)
        q, k = np.abs(q), -np.abs(k) * 1e3
        scale, block = 1.0, 8
    else:
        q, k, v = _rand(1, 1, 64, 8, 32)
        scale, block = 0.35, 8
    O, L = oracle_mod.attention_fwd(q, k, v, scale, False)
    good = oracle_mod.online_merge(q[0, 0], k[0, 0], v[0, 0], scale, False, block)
    bad = oracle_mod.online_merge(q[0, 0], k[0, 0], v[0, 0], scale, False, block, mutation=mutation)
    assert _worst(np.abs(good[0] - O[0, 0]).max(), np.abs(good[1] - L[0, 0]).max()) < TOL
    diff = np.abs(np.nan_to_num(bad[0], nan=1e9) - O[0, 0]).max()
    diff = max(diff, np.abs(np.nan_to_num(bad[1], nan=1e9, posinf=1e9) - L[0, 0]).max())
    assert diff > 1e-3


# ------------------------------------------------ mutants of the C oracle itself
MUTANTS = {
    "scale dropped": ("const double s = jb->scale * dot;", "const double s = dot;"),
    "causal off by one": ("nvis = (i + 1 < n) ? i + 1 : n;", "nvis = (i < n) ? i : n;"),
    "K indexed by query row": ("const double *kj = jb->k + j * d;", "const double *kj = jb->k + i * d;"),
    "K transposed stride": ("const double *kj = jb->k + j * d;", "const double *kj = jb->k + j;"),
    "wrong exp sign": ("exp(jb->scores[j] - m)", "exp(m - jb->scores[j])"),
    "missing normalisation": ("o_row[c] /= l;", "o_row[c] /= 1.0;"),
    "LSE without max": ("*lse_out = m + log(l);", "*lse_out = log(l);"),
    "LSE in log2": ("*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    "V indexed by query row": ("const double *vj = jb->v + j * d;", "const double *vj = jb->v + i * d;"),
    "max not tracked": ("if (s > m) m = s;", "m = 0.0;"),
    "weights not summed": ("l += w;", "l = w;"),
    "one key dropped": ("for (long j = 0; j < nvis; ++j) {\n        const double w", "for (long j = 1; j < nvis; ++j) {\n        const double w"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_oracle_mutants(oracle_mod, tmp_path, name):
    src_path = os.path.join(os.path.dirname(oracle_mod.__file__), "fa2_oracle.c")
    src = open(src_path).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "mutant.c"
    so_path = tmp_path / "libmutant.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", str(c_path), "-o",
                    str(so_path), "-lm"], check=True)
    attn = _attn(oracle_mod, libpath=str(so_path))
    failed = []
    for pin in PINS:
        try:
            err = pin(attn)
        except Exception:
            err = float("inf")
        if not (err < TOL):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the mutant '{name}'"


# ------------------------------------------------------------------ workloads
def test_workload_inputs_are_seeded_and_shaped():
    w = workloads.WORKLOADS["ragged"]
    small = workloads.custom(w.B, w.H, 64, w.D, w.dtype, seed=w.seed, sigma_qk=3.0)
    a = workloads.make_inputs(small)
    b = workloads.make_inputs(small)
    for x, y in zip(a, b):
        assert torch.equal(x, y) and x.dtype == torch.float16 and x.shape == (2, 12, 64, 64)
    assert 2.5 < float(a[0].float().std()) < 3.5 and 0.8 < float(a[2].float().std()) < 1.2


def test_metric_flops_match_the_pages_table():
    """The pages' RTX 4090 table: the metric 4*B*H*N^2*D over the printed times gives the
    restated TFLOPS, and the page's own column follows B*H*N^2*(4D+5)."""
    with open(os.path.join(GOLDEN, "pages_perf_table.json")) as fh:
        tab = json.load(fh)
    w = workloads.WORKLOADS["pages"]
    assert (w.B, w.H, w.N, w.D) == (tab["B"], tab["H"], tab["N"], tab["D"])
    for row in tab["rows"]:
        t = row["ms"] * 1e-3
        assert abs(workloads.flops(w) / t / 1e12 - row["metric_tflops"]) < 0.051
        page = w.B * w.H * w.N ** 2 * (4 * w.D + 5) / t / 1e12
        assert abs(page - row["page_tflops"]) < 0.151


def test_flops_and_bytes_of_the_contract_workloads():
    W = workloads.WORKLOADS
    assert workloads.flops(W["tiny"]) == 4 * 128 * 128 * 64
    assert abs(workloads.flops(W["causal128"]) - 2.749e11) / 2.749e11 < 1e-3
    assert abs(workloads.flops(W["long"]) - 1.100e12) / 1.100e12 < 1e-3
    assert workloads.algorithmic_bytes(W["tiny"]) == 66048
    assert workloads.algorithmic_bytes(W["ragged"]) == 12384000
