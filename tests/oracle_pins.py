"""Pins that tie the CPU oracle to what the pages and the mathematics fix.

Each `pin_*` takes a loaded oracle library (so the same checks can run against deliberately
broken builds of the oracle, see test_oracle_mutants.py) and raises AssertionError on a
mismatch.  Sources of truth, none of them the oracle itself:
  * hand-worked dyadic cases (tests/golden/hand_cases.json, derived from section I.1 of the
    llmgo page, "Verification via Modified Rejection Sampling");
  * closed forms: V=2 softmax is a logistic function; residual mass = 1 - sum min(p, q);
  * library routines on special cases: numpy argmax (first occurrence), scipy softmax,
    numpy float16 / bit-shift bf16 widening;
  * brute force over tiny inputs (inverse CDF, tree paths);
  * the invariance theorem (section I.1, last paragraph) by chi-squared tests.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_cases.json")
TOL = oracle.DEFAULT_TOL


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ------------------------------------------------------------------------- hand cases ----
def pin_hand_chain_cases(lib):
    for case in _golden()["chain"]:
        p = np.asarray(case["p"], np.float64)
        K = p.shape[0] - 1
        q = np.asarray(case["q"], np.float64).reshape(K, p.shape[1])
        for run in case["runs"]:
            o = oracle.verify_probs(p, q, case["x"], run["r"], run["u"], TOL, lib=lib)
            tag = f"{case['name']} r={run['r']} u={run['u']}"
            assert int(o["num_accepted"]) == run["n_acc"], (tag, o)
            assert list(o["out_tokens"]) == run["out_tokens"], (tag, o)
            assert np.allclose(o["alpha"], case["alpha"], rtol=0, atol=1e-15), (tag, o["alpha"])
            assert np.allclose(o["mass"], case["mass"], rtol=0, atol=1e-15), (tag, o["mass"])
            assert bool(o["req_flag"] & oracle.FLAG_ACCEPT_TIE) == run["accept_tie"], (tag, o)
            assert bool(o["req_flag"] & oracle.FLAG_CDF_TIE) == run["cdf_tie"], (tag, o)
            assert bool(o["req_flag"] & oracle.FLAG_CDF_TIE_WIDE) == run.get("cdf_tie_wide", False), (tag, o)
            if "cand" in run:
                assert list(o["cand"]) == run["cand"], (tag, o["cand"])
                zr = [bool(f & oracle.FLAG_ZERO_RESIDUAL) for f in o["pos_flag"]]
                assert zr == run["zero_residual"], (tag, o["pos_flag"])


def pin_hand_tree_cases(lib):
    for case in _golden()["tree"]:
        o = oracle.tree_walk(case["parents"], case["tokens"], case["amax"], lib=lib)
        assert o["accept_len"] == case["accept_len"], (case["name"], o)
        assert list(o["path"]) == case["path"], (case["name"], o)
        assert list(o["out_tokens"]) == case["out_tokens"], (case["name"], o)
        v, d = oracle.tree_bruteforce(case["parents"], case["tokens"], case["amax"], lib=lib)
        assert d == case["accept_len"] and (d == 0 or v == case["path"][d]), (case["name"], v, d)


# ------------------------------------------------------------------------------ softmax ----
def pin_softmax_closed_forms(lib):
    # V = 2 reduces to the logistic function of the logit gap over T.
    for a, b, T in [(0.0, 1.0, 1.0), (1.5, -2.0, 0.7), (3.0, 3.5, 2.0), (-7.0, 9.0, 0.25)]:
        p, e = oracle.softmax([a, b], T, lib=lib)
        assert e == 0
        want1 = 1.0 / (1.0 + math.exp(-(b - a) / T))
        assert abs(p[1] - want1) < 1e-15 and abs(p[0] - (1 - want1)) < 1e-15, (a, b, T, p)
    # Equal logits give the uniform distribution for any T.
    p, _ = oracle.softmax(np.full(7, 2.5), 0.3, lib=lib)
    assert np.allclose(p, 1 / 7, atol=1e-16)
    # Temperature divides the logits: softmax(l, T) == softmax(l / T, 1).
    rng = np.random.default_rng(1)
    l = rng.normal(0, 3, 50)
    p1, _ = oracle.softmax(l, 0.7, lib=lib)
    p2, _ = oracle.softmax(l / 0.7, 1.0, lib=lib)
    assert np.allclose(p1, p2, rtol=1e-13, atol=0)
    # Shift invariance and normalisation.
    p3, _ = oracle.softmax(l + 123.0, 0.7, lib=lib)
    assert np.allclose(p1, p3, rtol=1e-12, atol=0)
    assert abs(p1.sum() - 1.0) < 1e-12
    # Library routine on the same row.
    from scipy.special import softmax as sp_softmax

    assert np.allclose(p1, sp_softmax(l / 0.7), rtol=1e-12, atol=1e-300)
    # -inf is a masked token with probability 0; NaN / +inf / all -inf are errors.
    p4, e4 = oracle.softmax([0.0, -np.inf, 0.0], 1.0, lib=lib)
    assert e4 == 0 and p4[1] == 0.0 and abs(p4[0] - 0.5) < 1e-16
    for bad in ([0.0, np.nan], [0.0, np.inf], [-np.inf, -np.inf]):
        assert oracle.softmax(bad, 1.0, lib=lib)[1] == oracle.ERR_NONFINITE


def pin_argmax_first_occurrence(lib):
    rng = np.random.default_rng(2)
    for _ in range(200):
        l = rng.integers(-3, 4, size=rng.integers(1, 40)).astype(np.float64)  # many ties
        assert oracle.argmax(l, lib=lib) == int(np.argmax(l))
    assert oracle.argmax([-0.0, 0.0, -1.0], lib=lib) == 0  # -0 == +0: lowest index
    assert oracle.argmax([-np.inf, -np.inf], lib=lib) == 0


# -------------------------------------------------------------------------- inverse CDF ----
def _brute_inverse_cdf(w, u):
    """The definition with exact rational arithmetic on dyadic weights."""
    from fractions import Fraction

    W = [Fraction(x) for x in w]
    S = sum(W)
    t = Fraction(u) * S
    C = Fraction(0)
    for i, x in enumerate(W):
        C += x
        if C > t:
            return i
    return max(i for i, x in enumerate(W) if x > 0)


def pin_inverse_cdf_definition(lib):
    rng = np.random.default_rng(3)
    for _ in range(300):
        V = int(rng.integers(1, 12))
        w = rng.integers(0, 5, size=V).astype(np.float64) / 8.0  # dyadic, zeros included
        if w.sum() == 0:
            w[rng.integers(V)] = 0.125
        for u in [0.0, 0.25, 0.5, float(rng.integers(0, 1 << 24)) / (1 << 24), 1 - 2**-24]:
            i, S, _ = oracle.inverse_cdf(w, u, lib=lib)
            assert i == _brute_inverse_cdf(w, u), (w, u, i)
            assert w[i] > 0  # a zero-weight token is never drawn
            assert S == w.sum()
    assert oracle.inverse_cdf(np.zeros(4), 0.5, lib=lib)[0] == -1


def pin_inverse_cdf_frequencies(lib):
    """On a grid of u the draw frequencies equal the normalised weights (up to grid size)."""
    w = np.array([0.0, 3.0, 1.0, 0.0, 4.0])
    n = 4096
    counts = np.zeros(w.size)
    for j in range(n):
        counts[oracle.inverse_cdf(w, (j + 0.5) / n, lib=lib)[0]] += 1
    assert np.allclose(counts / n, w / w.sum(), atol=1.0 / n)


# ---------------------------------------------------------------- residual closed forms ----
def _rand_dist(rng, V, sigma=2.0):
    l = rng.normal(0, sigma, V)
    e = np.exp(l - l.max())
    return e / e.sum()


def pin_residual_mass_closed_form(lib):
    rng = np.random.default_rng(4)
    for _ in range(50):
        V, K = int(rng.integers(2, 30)), int(rng.integers(1, 6))
        p = np.stack([_rand_dist(rng, V) for _ in range(K + 1)])
        q = np.stack([_rand_dist(rng, V) for _ in range(K)])
        x = rng.integers(0, V, K)
        o = oracle.verify_probs(p, q, x, np.full(K, 0.5, np.float32), 0.5, lib=lib)
        for k in range(K):
            tv = 1.0 - np.minimum(p[k], q[k]).sum()  # total-variation distance
            assert abs(o["mass"][k] - tv) < 1e-12, (k, o["mass"][k], tv)
            want = min(1.0, p[k, x[k]] / q[k, x[k]])
            assert abs(o["alpha"][k] - want) < 1e-15
        assert abs(o["mass"][K] - 1.0) < 1e-12


def pin_ngram_general_equals_shortcut(lib):
    rng = np.random.default_rng(5)
    for _ in range(100):
        V, K = int(rng.integers(2, 40)), int(rng.integers(1, 7))
        p = np.stack([_rand_dist(rng, V, 3.0) for _ in range(K + 1)])
        x = rng.integers(0, V, K)
        q = np.zeros((K, V))
        q[np.arange(K), x] = 1.0
        r = ((rng.integers(0, 1 << 24, K) + 1) / (1 << 24)).astype(np.float32)
        u = np.float32(rng.integers(0, 1 << 24) / (1 << 24))
        g = oracle.verify_probs(p, q, x, r, u, lib=lib)
        d = oracle.verify_ngram_direct(p, x, r, u, lib=lib)
        for key in ("num_accepted", "out_tokens", "cand"):
            assert np.array_equal(g[key], d[key]), key
        # the draft-model path widens its residual tie band to tol / S: its flags contain the
        # shortcut's
        assert np.all((g["pos_flag"] & d["pos_flag"]) == d["pos_flag"])
        assert (g["req_flag"] & d["req_flag"]) == d["req_flag"]
        assert np.array_equal(g["alpha"], d["alpha"]) and np.array_equal(g["mass"], d["mass"])
        assert np.allclose(g["alpha"], p[np.arange(K), x], atol=0)  # alpha = p(x) for one-hot q


def pin_ngram_on_logits(lib):
    """The logits-level n-gram call (explicit one-hot q) equals the shortcut on library softmax."""
    from scipy.special import softmax as sp_softmax

    rng = np.random.default_rng(10)
    B, K, V, T = 40, 4, 33, np.float32(0.8)
    lt = rng.normal(0, 3, (B, K + 1, V)).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    lt[np.arange(B)[:, None], np.arange(K)[None, :], x] += 4.0
    r = ((rng.integers(0, 1 << 24, (B, K)) + 1) / (1 << 24)).astype(np.float32)
    u = (rng.integers(0, 1 << 24, B) / (1 << 24)).astype(np.float32)
    o = oracle.verify_ngram("f32", lt, B, K, V, T, x, r, u, lib=lib)
    for b in range(B):
        p = sp_softmax(lt[b].astype(np.float64) / float(T), axis=-1)
        d = oracle.verify_ngram_direct(p, x[b], r[b], u[b], lib=lib)
        assert np.allclose(o["alpha"][b], d["alpha"], rtol=1e-12, atol=0)
        assert np.allclose(o["mass"][b], d["mass"], rtol=1e-10, atol=1e-15)
        if not d["req_flag"]:
            assert o["num_accepted"][b] == d["num_accepted"]
            assert np.array_equal(o["out_tokens"][b], d["out_tokens"])


# ------------------------------------------------------------------------------ greedy ----
def pin_greedy_chain(lib):
    rng = np.random.default_rng(6)
    for _ in range(100):
        K, V = int(rng.integers(0, 6)), int(rng.integers(1, 20))
        lt = rng.integers(-2, 3, size=(1, K + 1, V)).astype(np.float32)  # ties on purpose
        a = np.argmax(lt[0], axis=-1)
        x = np.where(rng.random(K) < 0.7, a[:K], rng.integers(0, V, K)).astype(np.int32)
        o = oracle.verify_chain("f32", lt, None, 1, K, V, 0.0, x[None], None, None, lib=lib)
        n = 0
        while n < K and x[n] == a[n]:
            n += 1
        assert o["num_accepted"][0] == n
        want = list(x[:n]) + [a[n]] + [-1] * (K - n)
        assert list(o["out_tokens"][0]) == want
        assert o["err"][0] == 0


def pin_greedy_is_low_temperature_limit(lib):
    """T -> 0 makes p one-hot; with a greedy draft the sampled call equals the greedy call."""
    rng = np.random.default_rng(7)
    for _ in range(40):
        K, V = 4, 16
        lt = rng.normal(0, 3, (1, K + 1, V)).astype(np.float32)
        ld = lt[:, :K] + rng.normal(0, 1, (1, K, V)).astype(np.float32)
        x = np.argmax(ld, -1).astype(np.int32)
        r = np.full((1, K), 0.5, np.float32)
        u = np.full(1, 0.5, np.float32)
        g = oracle.verify_chain("f32", lt, ld, 1, K, V, 0.0, x, r, u, lib=lib)
        s = oracle.verify_chain("f32", lt, ld, 1, K, V, 1e-4, x, r, u, lib=lib)
        assert np.array_equal(g["out_tokens"], s["out_tokens"]), (g, s)
        assert np.array_equal(g["num_accepted"], s["num_accepted"])


# --------------------------------------------------------------------- input widening ----
def pin_input_widening(lib):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f16 = h.view(np.float16).astype(np.float64)
    got = oracle.load_elems(h, "f16", lib=lib)
    fin = np.isfinite(f16)
    assert np.array_equal(got[fin], f16[fin]) and np.array_equal(np.isnan(got), np.isnan(f16))
    with np.errstate(invalid="ignore"):
        bf = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = oracle.load_elems(h, "bf16", lib=lib)
    fin = np.isfinite(bf)
    assert np.array_equal(got[fin], bf[fin]) and np.array_equal(np.isnan(got), np.isnan(bf))


# ------------------------------------------------------------------------- error bits ----
def pin_error_semantics(lib):
    K, V = 2, 5
    rng = np.random.default_rng(8)
    lt = rng.normal(0, 1, (3, K + 1, V)).astype(np.float32)
    ld = rng.normal(0, 1, (3, K, V)).astype(np.float32)
    x = np.array([[0, 1], [0, V], [1, 2]], np.int32)  # request 1 has an out-of-range token
    lt[2, 1, 3] = np.nan  # request 2 has a NaN target logit
    r = np.full((3, K), 0.5, np.float32)
    u = np.full(3, 0.5, np.float32)
    o = oracle.verify_chain("f32", lt, ld, 3, K, V, 1.0, x, r, u, lib=lib)
    assert list(o["err"]) == [0, oracle.ERR_BAD_TOKEN, oracle.ERR_NONFINITE]
    for b in (1, 2):
        assert o["num_accepted"][b] == 0 and (o["out_tokens"][b] == -1).all()
    g = oracle.verify_chain("f32", lt, None, 3, K, V, 0.0, x, None, None, lib=lib)
    assert list(g["err"]) == [0, oracle.ERR_BAD_TOKEN, oracle.ERR_NONFINITE]


# ---------------------------------------------------------------------------- trees ----
def random_tree(rng, N1, V, distinct=True):
    parents = np.full(N1, -1, np.int32)
    tokens = np.zeros(N1, np.int32)
    for i in range(1, N1):
        parents[i] = rng.integers(0, i)
    for p in range(N1):
        kids = np.nonzero(parents == p)[0]
        if kids.size:
            if distinct and kids.size <= V:
                tokens[kids] = rng.choice(V, size=kids.size, replace=False)
            else:
                tokens[kids] = rng.integers(0, V, kids.size)
    return parents, tokens


def pin_tree_walk_vs_bruteforce(lib, n_trees=2000):
    rng = np.random.default_rng(9)
    for _ in range(n_trees):
        N1, V = int(rng.integers(1, 21)), 24  # V >= N1 keeps every sibling set distinct
        parents, tokens = random_tree(rng, N1, V)
        amax = rng.integers(0, V, N1).astype(np.int32)
        # bias toward long accepted paths: copy a child's token into its parent's argmax
        for i in range(1, N1):
            if rng.random() < 0.6:
                amax[parents[i]] = tokens[i]
        o = oracle.tree_walk(parents, tokens, amax, lib=lib)
        v, d = oracle.tree_bruteforce(parents, tokens, amax, lib=lib)
        assert o["accept_len"] == d, (parents, tokens, amax, o, v, d)
        if d:
            assert o["path"][d] == v
        # the path is a chain of parent links with matching tokens
        path = o["path"][: d + 1]
        for j in range(1, d + 1):
            assert parents[path[j]] == path[j - 1] and tokens[path[j]] == amax[path[j - 1]]
            assert o["out_tokens"][j - 1] == tokens[path[j]]
        assert o["out_tokens"][d] == amax[path[d]]


def pin_tree_check(lib):
    assert oracle.tree_check([-1, 0, 1], [0, 1, 2], 3, lib=lib) == 0
    assert oracle.tree_check([0, 0, 1], [0, 1, 2], 3, lib=lib) == oracle.ERR_BAD_TREE
    assert oracle.tree_check([-1, 2, 1], [0, 1, 2], 3, lib=lib) == oracle.ERR_BAD_TREE
    assert oracle.tree_check([-1, 0, 1], [0, 1, 3], 3, lib=lib) == oracle.ERR_BAD_TOKEN


# ------------------------------------------------------------------ invariance theorem ----
def chi2_pvalue(counts: np.ndarray, probs: np.ndarray, min_expected: float = 5.0) -> float:
    """Pearson chi-squared p-value, bins with expected count < min_expected merged."""
    from scipy.stats import chi2

    n = counts.sum()
    exp = probs * n
    order = np.argsort(exp)
    c_m, e_m, acc_c, acc_e = [], [], 0.0, 0.0
    for i in order:
        acc_c += counts[i]
        acc_e += exp[i]
        if acc_e >= min_expected:
            c_m.append(acc_c)
            e_m.append(acc_e)
            acc_c = acc_e = 0.0
    if acc_e > 0 and e_m:
        c_m[-1] += acc_c
        e_m[-1] += acc_e
    c_m, e_m = np.asarray(c_m), np.asarray(e_m)
    if c_m.size < 2:
        return 1.0
    stat = ((c_m - e_m) ** 2 / e_m).sum()
    return float(chi2.sf(stat, c_m.size - 1))


def invariance_check(out_tokens, n_acc, p_rows, K, alpha_min=1e-3):
    """At every position k, the token emitted there (by trials that reached k) follows p_k."""
    pvals = []
    for k in range(K + 1):
        reached = n_acc >= k
        toks = out_tokens[reached, k]
        counts = np.bincount(toks, minlength=p_rows.shape[1]).astype(np.float64)
        pv = chi2_pvalue(counts, p_rows[k])
        pvals.append(pv)
        assert pv > alpha_min, (k, pv, counts, p_rows[k] * counts.sum())
    return pvals


def acceptance_check(n_acc, p_rows, q_rows, K, sigmas=4.0):
    """P(accept at k | reached k) = sum_i min(p_k(i), q_k(i)); E[n_acc] = sum_k prod_{t<=k} beta_t."""
    beta = np.minimum(p_rows[:K], q_rows[:K]).sum(axis=1)
    for k in range(K):
        reached = (n_acc >= k).sum()
        acc = (n_acc > k).sum()
        sd = math.sqrt(reached * beta[k] * (1 - beta[k])) + 1e-9
        assert abs(acc - reached * beta[k]) <= sigmas * sd + 1, (k, acc, reached * beta[k], sd)
    expect = sum(np.prod(beta[: k + 1]) for k in range(K))
    sd = n_acc.std() / math.sqrt(n_acc.size)
    assert abs(n_acc.mean() - expect) <= sigmas * sd, (n_acc.mean(), expect, sd)
    return beta


FAST_PINS = [pin_hand_chain_cases, pin_hand_tree_cases, pin_softmax_closed_forms,
             pin_argmax_first_occurrence, pin_inverse_cdf_definition, pin_inverse_cdf_frequencies,
             pin_residual_mass_closed_form, pin_ngram_general_equals_shortcut, pin_ngram_on_logits,
             pin_greedy_chain,
             pin_greedy_is_low_temperature_limit, pin_input_widening, pin_error_semantics,
             pin_tree_check]


def pin_error_bits_accumulate(lib):
    """Reading R11: every applicable error bit is reported (a bad token and a NaN row together)."""
    K, V = 2, 6
    lt = np.zeros((1, K + 1, V), np.float32)
    lt[0, 2, 1] = np.nan
    ld = np.zeros((1, K, V), np.float32)
    x = np.array([[0, V + 3]], np.int32)
    r = np.full((1, K), 0.5, np.float32)
    u = np.full(1, 0.5, np.float32)
    both = oracle.ERR_BAD_TOKEN | oracle.ERR_NONFINITE
    assert oracle.verify_chain("f32", lt, ld, 1, K, V, 1.0, x, r, u, lib=lib)["err"][0] == both
    assert oracle.verify_chain("f32", lt, None, 1, K, V, 0.0, x, None, None, lib=lib)["err"][0] == both
    assert oracle.verify_ngram("f32", lt, 1, K, V, 1.0, x, r, u, lib=lib)["err"][0] == both


FAST_PINS.append(pin_error_bits_accumulate)


def pin_residual_band_scales_with_mass(lib):
    """Reading R10: the max(0, p - q) draw is flagged in the strict tier within tol of a CDF
    boundary, and in the widened tier within tol / S but not tol (tol when S = 1)."""
    p = np.array([[0.6, 0.4], [0.5, 0.5]])
    q = np.array([[0.5, 0.5]])  # residual [0.1, 0]: S = 0.1, C/S = [1, 1]
    x, r = [1], [0.9375]  # alpha = 0.8, rejected
    for u, strict, wide in [(2e-6, False, True), (9e-6, False, True), (5e-7, True, False),
                            (2e-5, False, False), (0.5, False, False)]:
        o = oracle.verify_probs(p, q, x, r, u, TOL, lib=lib)
        assert o["num_accepted"] == 0 and o["out_tokens"][0] == 0
        assert abs(o["mass"][0] - 0.1) < 1e-15
        assert bool(o["req_flag"] & oracle.FLAG_CDF_TIE) == strict, (u, o)
        assert bool(o["req_flag"] & oracle.FLAG_CDF_TIE_WIDE) == wide, (u, o)
    # disjoint supports: S = 1, the band stays tol and no widened tier exists
    p2 = np.array([[1.0, 0.0], [0.5, 0.5]])
    q2 = np.array([[0.0, 1.0]])
    o = oracle.verify_probs(p2, q2, [1], [0.5], 2e-6, TOL, lib=lib)
    assert not (o["req_flag"] & (oracle.FLAG_CDF_TIE | oracle.FLAG_CDF_TIE_WIDE))
    # the n-gram residual (p with x removed) takes no widened tier either
    o = oracle.verify_ngram_direct(np.array([[0.25, 0.75], [0.5, 0.5]]), [1], [0.9375], 2e-6, TOL, lib=lib)
    assert o["num_accepted"] == 0 and not (o["req_flag"] & oracle.FLAG_CDF_TIE_WIDE)


FAST_PINS.append(pin_residual_band_scales_with_mass)


# -------------------------------------------------------------- stochastic tree walk ----
def pin_hand_tree_sample_cases(lib):
    """Hand-worked walks (tests/golden/hand_cases.json, "tree_sample")."""
    for case in _golden()["tree_sample"]:
        p, q = np.asarray(case["p"], np.float64), np.asarray(case["q"], np.float64)
        for run in case["runs"]:
            o = oracle.tree_sample_probs(p, q, case["parents"], case["tokens"], run["r"], run["u"],
                                         TOL, lib=lib)
            tag = f"{case['name']} r={run['r']} u={run['u']}"
            assert o["accept_len"] == run["accept_len"], (tag, o)
            assert list(o["path"]) == run["path"], (tag, o)
            assert list(o["out_tokens"]) == run["out_tokens"], (tag, o)
            assert np.allclose(o["alpha"], run["alpha"], rtol=0, atol=1e-15), (tag, o["alpha"])
            assert abs(o["mass"] - run["mass"]) <= 1e-15, (tag, o["mass"])
            assert bool(o["req_flag"] & oracle.FLAG_ACCEPT_TIE) == run["accept_tie"], (tag, o)
            assert bool(o["req_flag"] & oracle.FLAG_CDF_TIE) == run["cdf_tie"], (tag, o)
            assert bool(o["req_flag"] & oracle.FLAG_ACCEPT_TIE_WIDE) == run.get("accept_tie_wide", False), (tag, o)
            assert bool(o["req_flag"] & oracle.FLAG_CDF_TIE_WIDE) == run.get("cdf_tie_wide", False), (tag, o)
            if "draw_w" in run:  # the final draw's weights, and their cumulative sums over the total
                assert np.allclose(o["draw_w"], run["draw_w"], rtol=0, atol=1e-15), (tag, o["draw_w"])
                assert np.allclose(o["draw_wmax"], run["draw_wmax"], rtol=0, atol=1e-12), (tag, o["draw_wmax"])
                w = np.asarray(run["draw_w"])
                assert np.allclose(o["draw_cdf"], np.cumsum(w) / w.sum(), rtol=0, atol=1e-15), (tag, o)
            f = oracle.tree_sample_probs(p, q, case["parents"], case["tokens"], run["r"], run["u"],
                                         TOL, lib=lib, flip=True)
            if "flipped" in run:  # the other decision of the flagged test, worked by hand
                alt = run["flipped"]
                assert f["accept_len"] == alt["accept_len"], (tag, f)
                assert list(f["path"]) == alt["path"] and list(f["out_tokens"]) == alt["out_tokens"], (tag, f)
                assert np.allclose(f["draw_w"], alt["draw_w"], rtol=0, atol=1e-15), (tag, f["draw_w"])
                assert np.allclose(f["draw_wmax"], alt["draw_wmax"], rtol=0, atol=1e-12), (tag, f["draw_wmax"])
                assert bool(f["req_flag"] & oracle.FLAG_CDF_TIE) == alt["cdf_tie"], (tag, f)
            elif not (run["accept_tie"] or run.get("accept_tie_wide", False)):  # nothing to flip
                assert f["accept_len"] == o["accept_len"] and list(f["out_tokens"]) == list(o["out_tokens"]), tag


def pin_tree_sample_chain_reduction(lib, n_cases=60):
    """A tree with one child per node is a chain: the walk must give the chain verification of
    section I.1 (pinned on its own) on the same rows, uniforms and tokens."""
    rng = np.random.default_rng(31)
    for i in range(n_cases):
        K, V = int(rng.integers(0, 6)), int(rng.integers(2, 12))
        T = float(rng.choice([0.5, 1.0, 1.7]))
        lt = (rng.normal(0, 2, (1, K + 1, V))).astype(np.float32)
        ld = (lt[:, :K] + rng.normal(0, 1, (1, K, V))).astype(np.float32)
        x = rng.integers(0, V, (1, K)).astype(np.int32)
        r = ((rng.integers(0, 1 << 24, (1, K)) + 1) / float(1 << 24)).astype(np.float32)
        if i % 3 == 0 and K:
            r[0, : K // 2 + 1] = np.float32(2.0 ** -24)  # long accepted prefixes too
        u = (rng.integers(0, 1 << 24, 1) / float(1 << 24)).astype(np.float32)
        ch = oracle.verify_chain("f32", lt, ld, 1, K, V, T, x, r, u, lib=lib)
        parents = np.arange(-1, K, dtype=np.int32)[None]
        tokens = np.concatenate([[[0]], x], axis=1).astype(np.int32)
        dt = np.concatenate([ld, np.zeros((1, 1, V), np.float32)], axis=1)  # the leaf's draft row
        rt = np.concatenate([[[1.0]], r], axis=1).astype(np.float32)
        tr = oracle.verify_tree_sample("f32", lt, dt, 1, K, V, T, tokens, parents, rt, u, lib=lib)
        n = int(ch["num_accepted"][0])
        assert tr["accept_len"][0] == n, (i, ch, tr)
        assert list(tr["out_tokens"][0]) == list(ch["out_tokens"][0]), (i, ch, tr)
        assert list(tr["path"][0][: n + 1]) == list(range(n + 1)) and (tr["path"][0][n + 1:] == -1).all()
        assert abs(tr["mass"][0] - (ch["mass"][0][n] if n < K else 1.0)) <= 1e-12, (i, ch, tr)
        # the children tested are the draft positions up to the rejected one
        assert np.allclose(tr["alpha"][0][1: min(n + 1, K) + 1], ch["alpha"][0][: min(n + 1, K)],
                           rtol=0, atol=1e-15)
        assert tr["req_flag"][0] == ch["req_flag"][0], (i, ch, tr)


def pin_tree_sample_residual_closed_form(lib, n_cases=200):
    """After j rejected siblings the target is max(0, p - c_j q) / R_j with c_1 = 0, R_1 = 1,
    c_{j+1} = c_j + R_j and R_j = sum_i max(0, p_i - c_j q_i): an identity derived from the
    residual step (max(0, max(0, p - c q) - R q) = max(0, p - (c + R) q) for q >= 0), checked on
    the alpha of every sibling, the mass and the drawn token."""
    rng = np.random.default_rng(47)
    for _ in range(n_cases):
        V, m = int(rng.integers(2, 10)), int(rng.integers(1, 6))
        p = _rand_dist(rng, V)
        q = _rand_dist(rng, V)
        toks = rng.integers(0, V, m)
        parents = np.array([-1] + [0] * m, np.int32)
        tokens = np.concatenate([[0], toks]).astype(np.int32)
        r = np.ones(m + 1, np.float32)  # accept only where alpha == 1
        u = float(rng.integers(0, 1 << 24) / float(1 << 24))
        P = np.vstack([p] + [p] * m)
        Q = np.vstack([q] + [q] * m)
        o = oracle.tree_sample_probs(P, Q, parents, tokens, r, u, TOL, lib=lib)
        c, R = 0.0, 1.0
        accepted = None
        for j, x in enumerate(toks, start=1):
            num = max(0.0, p[x] - c * q[x])
            a = 1.0 if (q[x] == 0 or num >= R * q[x]) else num / (R * q[x])
            assert abs(o["alpha"][j] - a) <= 1e-9 * max(1.0, a), (j, o["alpha"], a)
            if a >= 1.0:
                accepted = j
                break
            c, R = c + R, np.maximum(0.0, p - (c + R) * q).sum()
        if accepted is not None:
            assert o["accept_len"] == 1 and o["path"][1] == accepted
            continue
        w = np.maximum(0.0, p - c * q)
        assert abs(o["mass"] - R) <= 1e-9, (o["mass"], R)
        if o["req_flag"] & (oracle.FLAG_CDF_TIE | oracle.FLAG_ZERO_RESIDUAL):
            continue
        assert o["accept_len"] == 0 and o["out_tokens"][0] == _brute_inverse_cdf(w, u)


def pin_tree_sample_greedy_walk(lib, n_cases=300):
    """T == 0: the walk is the greedy tree walk (R9) of the pinned greedy tree verification."""
    rng = np.random.default_rng(53)
    for _ in range(n_cases):
        N1, V = int(rng.integers(1, 16)), 20
        parents, tokens = random_tree(rng, N1, V)
        lt = rng.normal(0, 1, (1, N1, V)).astype(np.float32)
        for i in range(1, N1):  # make matching paths likely
            if rng.random() < 0.6:
                lt[0, parents[i], tokens[i]] += 8.0
        g = oracle.verify_tree_greedy("f32", lt, 1, N1 - 1, V, tokens[None], parents[None], lib=lib)
        w = oracle.verify_tree_sample("f32", lt, None, 1, N1 - 1, V, 0.0, tokens[None],
                                      parents[None], None, None, lib=lib)
        assert w["accept_len"][0] == g["accept_len"][0]
        assert (w["path"][0] == g["path"][0]).all() and (w["out_tokens"][0] == g["out_tokens"][0]).all()
        assert w["err"][0] == 0 and w["mass"][0] == 1.0


def pin_tree_sample_errors(lib):
    """R11 and R14: a malformed tree or a bad token fails the request; a NaN row fails it only
    when the walk visits that node; a leaf's draft row is never read."""
    V, N = 4, 3
    parents = np.array([[-1, 0, 0, 1]], np.int32)
    tokens = np.array([[0, 1, 2, 3]], np.int32)
    lt = np.zeros((1, N + 1, V), np.float32)
    lt[0, 0, 2] = 9.0  # p_root concentrates on token 2: node 1 (token 1) rejected, node 2 accepted
    ld = np.zeros((1, N + 1, V), np.float32)
    ld[0, 2:] = np.nan  # leaves' draft rows: never read
    r = np.full((1, N + 1), 0.5, np.float32)
    u = np.full(1, 0.5, np.float32)
    o = oracle.verify_tree_sample("f32", lt, ld, 1, N, V, 1.0, tokens, parents, r, u, lib=lib)
    assert o["err"][0] == 0 and o["path"][0][1] == 2, o
    lt3 = lt.copy()
    lt3[0, 3, 0] = np.nan  # node 3 is not visited
    o = oracle.verify_tree_sample("f32", lt3, ld, 1, N, V, 1.0, tokens, parents, r, u, lib=lib)
    assert o["err"][0] == 0, o
    lt0 = lt.copy()
    lt0[0, 0, 1] = np.nan
    for T in (1.0, 0.0):
        o = oracle.verify_tree_sample("f32", lt0, ld, 1, N, V, T, tokens, parents, r, u, lib=lib)
        assert o["err"][0] == oracle.ERR_NONFINITE and o["accept_len"][0] == 0
        assert (o["out_tokens"][0] == -1).all() and (o["path"][0] == -1).all()
    ldr = np.zeros_like(ld)
    ldr[0, 0, 3] = np.inf
    o = oracle.verify_tree_sample("f32", lt, ldr, 1, N, V, 1.0, tokens, parents, r, u, lib=lib)
    assert o["err"][0] == oracle.ERR_NONFINITE
    bad = np.array([[-1, 0, 2, 1]], np.int32)
    o = oracle.verify_tree_sample("f32", lt, ld, 1, N, V, 1.0, tokens, bad, r, u, lib=lib)
    assert o["err"][0] == oracle.ERR_BAD_TREE
    o = oracle.verify_tree_sample("f32", lt, ld, 1, N, V, 1.0, np.array([[0, 1, 9, 3]], np.int32),
                                  parents, r, u, lib=lib)
    assert o["err"][0] == oracle.ERR_BAD_TOKEN


FAST_PINS += [pin_hand_tree_sample_cases, pin_tree_sample_chain_reduction,
              pin_tree_sample_residual_closed_form, pin_tree_sample_greedy_walk,
              pin_tree_sample_errors]


# ------------------------------------------------------------- prompt lookup drafting ----
def pin_hand_ngram_draft_cases(lib):
    for case in _golden()["ngram_draft"]:
        o = oracle.ngram_draft(np.asarray(case["ctx"], np.int32), case["K"], lib=lib)
        assert list(o["draft"]) == case["draft"], (case["name"], o)
        assert (o["draft_len"], o["match_n"], o["match_end"]) == (
            case["draft_len"], case["match_n"], case["match_end"]), (case["name"], o)


def _brute_ngram(ctx, K, n_max=4, n_min=1):
    """Every (n, end) pair whose n tokens before `end` equal the context's last n tokens, the best
    by (n, end); written independently of the oracle's loop order."""
    L = len(ctx)
    best = None
    for e in range(1, L):
        for n in range(n_min, n_max + 1):
            if n <= e and list(ctx[e - n:e]) == list(ctx[L - n:L]):
                if best is None or (n, e) > best:
                    best = (n, e)
    if best is None:
        return [-1] * K, 0, 0, -1
    n, e = best
    d = list(ctx[e:e + K])
    return d + [-1] * (K - len(d)), len(d), n, e


def pin_ngram_draft_bruteforce(lib, n_cases=3000):
    rng = np.random.default_rng(71)
    for _ in range(n_cases):
        L, Vs, K = int(rng.integers(0, 40)), int(rng.integers(1, 6)), int(rng.integers(1, 7))
        ctx = rng.integers(0, Vs, L).astype(np.int32)
        o = oracle.ngram_draft(ctx, K, lib=lib)
        d, ln, n, e = _brute_ngram(ctx, K)
        assert list(o["draft"]) == d and o["draft_len"] == ln, (ctx, K, o, d)
        assert (o["match_n"], o["match_end"]) == (n, e), (ctx, o, n, e)


def pin_ngram_draft_limits(lib):
    """n_max / n_min bound the n tried; the batched form equals the single form; a bad length."""
    ctx = np.array([1, 2, 3, 4, 0, 9, 1, 2, 3, 4], np.int32)
    assert oracle.ngram_draft(ctx, 3, n_max=4, lib=lib)["match_n"] == 4
    assert oracle.ngram_draft(ctx, 3, n_max=2, lib=lib)["match_n"] == 2
    assert oracle.ngram_draft(ctx, 3, n_max=4, n_min=4, lib=lib)["match_end"] == 4
    assert oracle.ngram_draft(np.array([1, 2, 1], np.int32), 3, n_min=2, lib=lib)["draft_len"] == 0
    rng = np.random.default_rng(5)
    ctxs = rng.integers(0, 4, (20, 30)).astype(np.int32)
    lens = rng.integers(0, 31, 20).astype(np.int32)
    lens[3] = 31  # longer than the array: invalid
    bo = oracle.ngram_draft_batch(ctxs, lens, 4, lib=lib)
    for b in range(20):
        if b == 3:
            assert bo["err"][b] == oracle.ERR_BAD_TOKEN and bo["draft_len"][b] == 0
            continue
        so = oracle.ngram_draft(ctxs[b, : lens[b]], 4, lib=lib)
        assert list(bo["draft"][b]) == list(so["draft"]) and bo["match_end"][b] == so["match_end"]


FAST_PINS += [pin_hand_ngram_draft_cases, pin_ngram_draft_bruteforce, pin_ngram_draft_limits]


# ---------------------------------------------------------- accepted-path KV compaction ----
def pin_hand_kv_compact_cases(lib):
    for case in _golden()["kv_compact"]:
        W, S = case["row_bytes"], len(case["slots"])
        cache = np.arange(S * W, dtype=np.uint8).reshape(S, W)
        out = oracle.kv_compact(cache, case["slots"], case["accept_len"], case["path"], lib=lib)
        assert out.tolist() == case["expected_rows"], (case["name"], out)
        ob, err = oracle.kv_compact_batch(cache[None], np.array([case["slots"]]), np.array([case["parents"]]),
                                          np.array([case["accept_len"]]), np.array([case["path"]]), lib=lib)
        assert err[0] == 0 and ob[0].tolist() == case["expected_rows"], case["name"]


def pin_kv_compact_sequential_moves(lib, n_cases=300):
    """Moving rows one at a time in increasing position, in place, gives the same cache: along an
    accepted path p_j >= j, so no move overwrites a row a later move still reads."""
    rng = np.random.default_rng(83)
    for _ in range(n_cases):
        N1, W = int(rng.integers(1, 30)), int(rng.integers(1, 9))
        parents, _tok = random_tree(rng, N1, 50)
        v = int(rng.integers(0, N1))
        path = [v]
        while path[-1] != 0:
            path.append(int(parents[path[-1]]))
        path = path[::-1]
        L = len(path) - 1
        slots = rng.permutation(N1 + 5)[:N1].astype(np.int32)
        cache = rng.integers(0, 256, (N1 + 5, W)).astype(np.uint8)
        pp = np.full(N1, -1, np.int32)
        pp[: L + 1] = path
        out = oracle.kv_compact(cache, slots, L, pp, lib=lib)
        seq = cache.copy()
        for j in range(1, L + 1):
            assert path[j] >= j
            seq[slots[j]] = seq[slots[path[j]]]
        assert np.array_equal(out, seq)
        moved = set(int(slots[j]) for j in range(1, L + 1))
        for srow in range(N1 + 5):
            if srow not in moved:
                assert np.array_equal(out[srow], cache[srow])


def pin_kv_compact_validation(lib):
    """A path that is not parent-linked, a length out of range or a slot out of range leaves the
    request untouched and flags it; the other requests of the batch are compacted."""
    parents = np.array([[-1, 0, 1, 1]] * 4, np.int32)
    slots = np.array([[0, 1, 2, 3], [4, 5, 6, 7], [8, 9, 10, 11], [12, 13, 14, 99]], np.int32)
    path = np.array([[0, 1, 3, -1], [0, 2, -1, -1], [0, 1, 3, -1], [0, 1, -1, -1]], np.int32)
    al = np.array([2, 1, 4, 1], np.int32)
    caches = np.arange(2 * 16 * 3, dtype=np.uint8).reshape(2, 16, 3)
    out, err = oracle.kv_compact_batch(caches, slots, parents, al, path, lib=lib)
    assert list(err) == [0, oracle.ERR_BAD_TREE, oracle.ERR_BAD_TREE, oracle.ERR_BAD_TREE]
    assert np.array_equal(out[:, 4:], caches[:, 4:])
    assert np.array_equal(out[:, 2], caches[:, 3]) and np.array_equal(out[:, 1], caches[:, 1])


FAST_PINS += [pin_hand_kv_compact_cases, pin_kv_compact_sequential_moves, pin_kv_compact_validation]


def pin_tree_walk_per_request_temperature(lib):
    """R18: a batch with one temperature per request (greedy ones included) gives, request by
    request, what a call at that request's temperature gives; a bad temperature fails only its
    request."""
    rng = np.random.default_rng(97)
    B, V = 8, 12
    par = np.array([-1, 0, 0, 1, 1, 2], np.int32)
    N1 = par.size
    lt = rng.normal(0, 2, (B, N1, V)).astype(np.float32)
    ld = (lt + rng.normal(0, 1, (B, N1, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, N1)).astype(np.int32)
    parents = np.broadcast_to(par, (B, N1)).copy()
    r = ((rng.integers(0, 1 << 24, (B, N1)) + 1) / float(1 << 24)).astype(np.float32)
    u = (rng.integers(0, 1 << 24, B) / float(1 << 24)).astype(np.float32)
    temps = np.array([0.5, 0.0, 1.0, 2.0, 0.0, 0.8, np.nan, -1.0], np.float32)
    o = oracle.verify_tree_sample("f32", lt, ld, B, N1 - 1, V, 1.0, tok, parents, r, u, lib=lib,
                                  temperatures=temps)
    for b in range(6):
        one = oracle.verify_tree_sample("f32", lt[b:b + 1], ld[b:b + 1], 1, N1 - 1, V, float(temps[b]),
                                        tok[b:b + 1], parents[b:b + 1], r[b:b + 1], u[b:b + 1], lib=lib)
        for k in ("accept_len", "path", "out_tokens", "alpha", "mass", "req_flag", "err"):
            assert np.array_equal(o[k][b], one[k][0]), (b, k)
    assert list(o["err"][6:]) == [oracle.ERR_BAD_TEMP] * 2 and (o["out_tokens"][6:] == -1).all()


FAST_PINS.append(pin_tree_walk_per_request_temperature)


def pin_chain_draw_rows(lib):
    """The draw rows given for checking flagged ties: at a draft position the step-3 residual
    max(0, p_k - q_k) of section I.1 (n-gram: p_k with x_k removed, q one-hot), at the bonus row
    p_K, and p_k itself where the residual is empty (R5), with p and q from scipy's softmax; the
    cdf is their cumulative sum over the total (numpy); and the inverse CDF over each row at u is
    the position's candidate in the verification call."""
    from scipy.special import softmax as sp_softmax

    rng = np.random.default_rng(61)
    for i in range(40):
        B, K, V = 2, int(rng.integers(0, 5)), int(rng.integers(2, 40))
        T = float(np.float32(rng.choice([0.6, 1.0, 1.5])))  # the temperature the calls take (fp32)
        lt = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
        ld = (lt[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
        if i % 4 == 0 and K:
            ld[1, 0] = lt[1, 0]  # q = p at a position: the residual is empty there
        x = rng.integers(0, V, (B, K)).astype(np.int32)
        r = ((rng.integers(0, 1 << 24, (B, K)) + 1) / float(1 << 24)).astype(np.float32)
        u = (rng.integers(0, 1 << 24, B) / float(1 << 24)).astype(np.float32)
        for ngram in (False, True):
            if ngram:
                o = oracle.verify_ngram("f32", lt, B, K, V, T, x, r, u, lib=lib)
            else:
                o = oracle.verify_chain("f32", lt, ld, B, K, V, T, x, r, u, lib=lib)
            for b in range(B):
                d = oracle.chain_draw_rows("f32", lt, ld, B, K, V, T, x, b, ngram=ngram, lib=lib)
                w, cdf, wmax = d["w"], d["cdf"], d["wmax"]
                assert d["err"] == 0
                p = sp_softmax(lt[b].astype(np.float64) / T, axis=-1)
                q = np.zeros((K, V))
                if ngram:
                    q[np.arange(K), x[b]] = 1.0
                else:
                    q = sp_softmax(ld[b].astype(np.float64) / T, axis=-1)
                for k in range(K + 1):
                    ref = np.maximum(0.0, p[k] - q[k]) if k < K else p[k]
                    empty = not ref.sum() > 0
                    if empty:
                        ref = p[k]
                    assert np.allclose(w[k], ref, rtol=0, atol=1e-12), (i, ngram, b, k)
                    if k < K and not ngram and not empty:
                        # the widened tier's largest weights: p and q each known to a relative tol / 2
                        wm = np.maximum(0.0, p[k] - q[k] + 0.5 * TOL * (p[k] + q[k]))
                        assert np.allclose(wmax[k], wm, rtol=0, atol=1e-12), (i, b, k)
                    else:
                        assert np.array_equal(wmax[k], w[k])
                    assert np.allclose(cdf[k], np.cumsum(w[k]) / w[k].sum(), rtol=0, atol=1e-12)
                    if not o["pos_flag"][b][k] & (oracle.FLAG_CDF_TIE | oracle.FLAG_CDF_TIE_WIDE):
                        assert o["cand"][b][k] == _brute_inverse_cdf(w[k], float(u[b])), (i, ngram, b, k)


FAST_PINS.append(pin_chain_draw_rows)


def pin_tree_sample_alt(lib):
    """The walk's outcome for one request without a flip is the walk itself (and its draw row is
    the last node's p, from scipy's softmax, when nothing was rejected there); with the first
    flagged accept test decided the other way it is, on a one-child tree, the chain verification
    (pinned on its own) with that position's r moved to the other side of alpha."""
    from scipy.special import softmax as sp_softmax

    rng = np.random.default_rng(67)
    done = 0
    for i in range(200):
        K, V = int(rng.integers(1, 6)), int(rng.integers(2, 12))
        T = float(np.float32(rng.choice([0.5, 1.0, 1.7])))
        lt = rng.normal(0, 2, (1, K + 1, V)).astype(np.float32)
        ld = (lt[:, :K] + rng.normal(0, 1, (1, K, V))).astype(np.float32)
        x = rng.integers(0, V, (1, K)).astype(np.int32)
        parents = np.arange(-1, K, dtype=np.int32)[None]
        tokens = np.concatenate([[[0]], x], axis=1).astype(np.int32)
        dt = np.concatenate([ld, np.zeros((1, 1, V), np.float32)], axis=1)
        u = (rng.integers(0, 1 << 24, 1) / float(1 << 24)).astype(np.float32)
        j = int(rng.integers(0, K))  # the position whose test is put on alpha
        rt = np.full((1, K + 1), 2.0 ** -24, np.float32)
        rt[0, j + 2:] = ((rng.integers(0, 1 << 24, K - j - 1) + 1) / float(1 << 24)).astype(np.float32)
        base = oracle.verify_tree_sample("f32", lt, dt, 1, K, V, T, tokens, parents, rt, u, lib=lib)
        a = float(base["alpha"][0][j + 1])
        if not (0.01 < a < 0.99):
            continue
        rt[0, j + 1] = np.float32(a)  # within tol of alpha: a flagged test
        o = oracle.verify_tree_sample("f32", lt, dt, 1, K, V, T, tokens, parents, rt, u, lib=lib)
        assert o["req_flag"][0] & oracle.FLAG_ACCEPT_TIE
        same = oracle.tree_sample_alt("f32", lt, dt, 1, K, V, T, tokens, parents, rt, u, 0, False, lib=lib)
        for k in ("accept_len", "mass", "req_flag"):
            assert same[k] == o[k][0], (i, k)
        assert list(same["out_tokens"]) == list(o["out_tokens"][0]) and list(same["path"]) == list(o["path"][0])
        L = same["accept_len"]
        if L == K or same["mass"] == 1.0:  # nothing rejected at the last node: the draw row is its p
            pl = sp_softmax(lt[0, L].astype(np.float64) / T)
            assert np.allclose(same["draw_w"], pl, rtol=0, atol=1e-12)
            assert np.array_equal(same["draw_wmax"], same["draw_w"])
            assert np.allclose(same["draw_cdf"], np.cumsum(pl) / pl.sum(), rtol=0, atol=1e-12)
        f = oracle.tree_sample_alt("f32", lt, dt, 1, K, V, T, tokens, parents, rt, u, 0, True, lib=lib)
        accepted = float(rt[0, j + 1]) <= a
        rc = rt[:, 1:].copy()
        rc[0, j] = np.float32(a + 1e-3) if accepted else np.float32(a - 1e-3)  # the other decision
        ch = oracle.verify_chain("f32", lt, ld, 1, K, V, T, x, rc, u, lib=lib)
        n = int(ch["num_accepted"][0])
        assert f["accept_len"] == n and n == (j if accepted else max(j + 1, n)), (i, f, ch)
        assert list(f["out_tokens"]) == list(ch["out_tokens"][0]), (i, f, ch)
        assert list(f["path"][: n + 1]) == list(range(n + 1))
        done += 1
    assert done >= 50, done


FAST_PINS.append(pin_tree_sample_alt)


def pin_chain_per_request_temperature(lib):
    """R18 on the chain and n-gram verification: a batch with one temperature per request (greedy
    ones included) gives, request by request, what a call at that request's temperature gives; a
    NaN, negative or infinite temperature fails its request alone, with the bad-temperature bit."""
    rng = np.random.default_rng(101)
    B, K, V = 9, 3, 14
    lt = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    ld = (lt[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    x[:, 0] = np.argmax(lt[:, 0], axis=-1)  # greedy requests accept their first draft
    r = ((rng.integers(0, 1 << 24, (B, K)) + 1) / float(1 << 24)).astype(np.float32)
    u = (rng.integers(0, 1 << 24, B) / float(1 << 24)).astype(np.float32)
    temps = np.array([0.5, 0.0, 1.0, 2.0, 0.0, 0.8, np.nan, -1.0, np.inf], np.float32)
    for ngram in (False, True):
        if ngram:
            o = oracle.verify_ngram("f32", lt, B, K, V, 1.0, x, r, u, lib=lib, temperatures=temps)
        else:
            o = oracle.verify_chain("f32", lt, ld, B, K, V, 1.0, x, r, u, lib=lib, temperatures=temps)
        for b in range(6):
            s = slice(b, b + 1)
            if ngram:
                one = oracle.verify_ngram("f32", lt[s], 1, K, V, float(temps[b]), x[s], r[s], u[s], lib=lib)
            else:
                one = oracle.verify_chain("f32", lt[s], ld[s], 1, K, V, float(temps[b]), x[s], r[s], u[s],
                                          lib=lib)
            for k in ("num_accepted", "out_tokens", "alpha", "cand", "mass", "pos_flag", "req_flag", "err"):
                assert np.array_equal(o[k][b], one[k][0]), (ngram, b, k)
        assert o["num_accepted"][1] >= 1 and o["num_accepted"][4] >= 1  # greedy: argmax drafts accepted
        assert list(o["err"][6:]) == [oracle.ERR_BAD_TEMP] * 3
        assert (o["out_tokens"][6:] == -1).all() and (o["num_accepted"][6:] == 0).all()


FAST_PINS.append(pin_chain_per_request_temperature)
