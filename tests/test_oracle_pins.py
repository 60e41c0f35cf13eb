"""The oracle against its pins: hand-worked cases, closed forms, library routines on special
cases, brute force, and the invariance theorem (chi-squared)."""

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

import oracle
import oracle_pins as pins
from speculative_decoding_verification_82_gb300 import synth


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", pins.FAST_PINS, ids=lambda f: f.__name__)
def test_fast_pin(pin, lib):
    pin(lib)


def test_tree_walk_equals_bruteforce(lib):
    pins.pin_tree_walk_vs_bruteforce(lib, n_trees=10_000)


def test_tree_duplicate_siblings_lowest_index(lib):
    # Reading R9: with duplicate sibling tokens the walk takes the lowest node index.
    parents = [-1, 0, 0, 1, 2]
    tokens = [0, 5, 5, 6, 7]
    amax = [5, 6, 7, 1, 2]
    o = oracle.tree_walk(parents, tokens, amax, lib=lib)
    assert o["accept_len"] == 2 and list(o["path"][:3]) == [0, 1, 3]
    assert list(o["out_tokens"][:3]) == [5, 6, 1]


def test_tree_greedy_on_logits_forced_path(lib):
    """Boosting the draft tokens of one root-to-leaf path makes exactly that path accepted."""
    rng = np.random.default_rng(11)
    parents = synth.eagle_tree_parents()
    N1, V = parents.size, 64
    for _ in range(20):
        tokens = np.zeros(N1, np.int32)
        for p in range(N1):
            kids = np.nonzero(parents == p)[0]
            if kids.size:
                tokens[kids] = rng.choice(V, kids.size, replace=False)
        leaf = int(rng.choice([i for i in range(N1) if not (parents == i).any()]))
        chain = []
        v = leaf
        while v != 0:
            chain.append(v)
            v = parents[v]
        chain = chain[::-1]
        lt = rng.normal(0, 1, (1, N1, V)).astype(np.float32)
        for v in chain:
            lt[0, parents[v], tokens[v]] += 50.0
        o = oracle.verify_tree_greedy("f32", lt, 1, N1 - 1, V, tokens[None], parents[None], lib=lib)
        assert o["err"][0] == 0
        assert o["accept_len"][0] == len(chain)
        assert list(o["path"][0][1:len(chain) + 1]) == chain
        assert o["out_tokens"][0][len(chain)] == np.argmax(lt[0, leaf])


def _run_tiny(lib, seed, trials, V, K=5):
    ci = synth.chain_tiny(seed=seed, trials=trials, K=K, V=V)
    o = oracle.verify_chain("f32", ci.target, ci.draft, ci.B, K, V, float(ci.temperature),
                            ci.draft_tokens, ci.r, ci.u, threads=8, lib=lib)
    T = float(ci.temperature)
    p = sp_softmax(ci.meta["target_rows"].astype(np.float64) / T, axis=-1)
    q = sp_softmax(ci.meta["draft_rows"].astype(np.float64) / T, axis=-1)
    return o, p, q


def test_invariance_theorem_v8_1e6_trials(lib):
    """Section I.1, invariance theorem: with x_k ~ q_k, the emitted token at every position
    follows p_k.  10^6 seeded trials at V=8, K=5, chi-squared per position."""
    K, V = 5, 8
    outs, nacc = [], []
    for s in range(4):
        o, p, q = _run_tiny(lib, 100 + s, 250_000, V, K) if s == 0 else _run_tiny_same(lib, s, V, K)
        outs.append(o["out_tokens"])
        nacc.append(o["num_accepted"])
        if s == 0:
            p0, q0 = p, q
    out = np.concatenate(outs)
    n = np.concatenate(nacc)
    pins.invariance_check(out, n, p0, K)
    pins.acceptance_check(n, p0, q0, K)


def _run_tiny_same(lib, s, V, K):
    """More trials on the same logits (seed 100): fresh draft tokens, r and u from other keys."""
    base = synth.chain_tiny(seed=100, trials=1, K=K, V=V)
    trials = 250_000
    rng = np.random.Generator(np.random.Philox(key=9000 + s))
    T = float(base.temperature)
    q = sp_softmax(base.meta["draft_rows"].astype(np.float64) / T, axis=-1)
    cq = np.cumsum(q, axis=-1)
    x = np.stack([np.minimum(np.searchsorted(cq[k], rng.random(trials), side="right"), V - 1)
                  for k in range(K)], axis=1).astype(np.int32)
    r = ((rng.integers(0, 1 << 24, (trials, K)) + 1) * synth.U24).astype(np.float32)
    u = (rng.integers(0, 1 << 24, trials) * synth.U24).astype(np.float32)
    target = np.broadcast_to(base.target[0], (trials, K + 1, V))
    draft = np.broadcast_to(base.draft[0], (trials, K, V))
    o = oracle.verify_chain("f32", target, draft, trials, K, V, T, x, r, u, threads=8, lib=lib)
    p = sp_softmax(base.meta["target_rows"].astype(np.float64) / T, axis=-1)
    return o, p, q


def test_invariance_theorem_chain_tiny_1e5_trials(lib):
    """Workload 1 (B=1, K=5, V=32, T=1): 10^5 seeded trials, chi-squared per position."""
    o, p, q = _run_tiny(lib, 0, 100_000, 32)
    pins.invariance_check(o["out_tokens"], o["num_accepted"], p, 5)
    pins.acceptance_check(o["num_accepted"], p, q, 5)
    flagged = (o["req_flag"] & (oracle.FLAG_ACCEPT_TIE | oracle.FLAG_CDF_TIE)) != 0
    assert flagged.mean() < 1e-3  # ties within 1e-6 are rare


def test_chi2_detects_a_wrong_distribution():
    """The chi-squared check itself has power: the draft distribution q instead of p fails."""
    rng = np.random.default_rng(12)
    p = sp_softmax(rng.normal(0, 2, 8))
    q = sp_softmax(np.log(p) + rng.normal(0, 1, 8))
    toks = np.searchsorted(np.cumsum(q), rng.random(100_000), side="right").clip(0, 7)
    counts = np.bincount(toks, minlength=8).astype(float)
    assert pins.chi2_pvalue(counts, p) < 1e-6


def test_invariance_theorem_tree_walk(lib):
    """Stochastic tree walk (each rejected sibling replaces the target by its residual): with
    children drawn independently from the parent's draft row, the token emitted after a prefix
    follows the target row of that prefix.  2 x 10^5 seeded trials at V=8, tree 1-3-6;
    chi-squared per prefix (root; each first token; each pair of first tokens with enough
    trials)."""
    ti = synth.tree_sample_tiny(seed=5, trials=200_000)
    T = float(ti.temperature)
    o = oracle.verify_tree_sample("f32", ti.target, ti.draft, ti.B, ti.N, ti.V, T, ti.node_tokens,
                                  ti.parents, ti.r, ti.u, threads=8, lib=lib)
    assert (o["err"] == 0).all()
    L, out = o["accept_len"], o["out_tokens"]
    p0 = sp_softmax(ti.meta["t0"].astype(np.float64) / T)
    p1 = sp_softmax(ti.meta["t1"].astype(np.float64) / T, axis=-1)
    p2 = sp_softmax(ti.meta["t2"].astype(np.float64) / T, axis=-1)
    V = ti.V
    assert pins.chi2_pvalue(np.bincount(out[:, 0], minlength=V).astype(float), p0) > 1e-3
    tested = 0
    for a in range(V):
        sel = (L >= 1) & (out[:, 0] == a)
        if sel.sum() >= 400:
            pv = pins.chi2_pvalue(np.bincount(out[sel, 1], minlength=V).astype(float), p1[a])
            assert pv > 1e-4, (a, pv)
            tested += 1
        for b in range(V):
            sel2 = (L >= 2) & (out[:, 0] == a) & (out[:, 1] == b)
            if sel2.sum() >= 400:
                pv = pins.chi2_pvalue(np.bincount(out[sel2, 2], minlength=V).astype(float), p2[a, b])
                assert pv > 1e-4, (a, b, pv)
                tested += 1
    assert tested >= 10
    # more than one sibling is tested in a good share of the walks (the residual update matters)
    assert ((o["alpha"][:, 2:4] >= 0).any(axis=1)).mean() > 0.2


def test_chi2_detects_a_tree_walk_without_residual_update(lib, tmp_path):
    """The tree invariance check has power: an oracle copy whose siblings are all tested against
    the node's own p (no residual update) fails it."""
    src = open(oracle.SRC).read()
    bad = src.replace("p[i] = w[i] / S;", "p[i] = p[i];")
    assert bad != src
    f = tmp_path / "mut.c"
    f.write_text(bad)
    mlib = oracle.load(oracle.build(str(f), str(tmp_path / "mut.so")))
    ti = synth.tree_sample_tiny(seed=5, trials=100_000)
    T = float(ti.temperature)
    o = oracle.verify_tree_sample("f32", ti.target, ti.draft, ti.B, ti.N, ti.V, T, ti.node_tokens,
                                  ti.parents, ti.r, ti.u, threads=8, lib=mlib)
    p0 = sp_softmax(ti.meta["t0"].astype(np.float64) / T)
    assert pins.chi2_pvalue(np.bincount(o["out_tokens"][:, 0], minlength=ti.V).astype(float), p0) < 1e-6


def test_ngram_lookup_reproduces_the_workload_drafts(lib):
    """The n-gram workload's drafts are the continuations of seeded prompt 4-grams; prompt lookup
    on the matching contexts (prompt + that 4-gram) proposes exactly them (a 4-gram repeat in a
    2048-token uniform prompt over 151936 tokens has probability below 1e-8)."""
    ctx, lens = synth.ngram_contexts(seed=0)
    o = oracle.ngram_draft_batch(ctx, lens, 5, threads=8, lib=lib)
    ng = synth.ngram(seed=0, B=256, V=151936)
    assert (o["match_n"] == 4).all() and (o["draft_len"] == 5).all()
    assert np.array_equal(o["draft"], ng.draft_tokens)
