"""GPU parity of the tree walk (spec_verify_tree_walk) against the CPU oracle on seeded inputs.

Stochastic walks (T > 0): the invariance check on the CUDA path (V = 8, tree 1-3-6), random
trees over the vocabulary sizes that select every cluster size (1 to 16 CTAs), the three element
types, ragged and misaligned rows, the EAGLE-2-like benchmark tree at V = 128256, more requests
than clusters resident at once, extreme temperatures.  Greedy walks (T = 0): against the oracle and
against spec_verify_tree_greedy (which reads every row).  Edge cases: the root alone, malformed
trees and tokens, non-finite visited rows, non-finite rows the walk never reads.  Per-request
temperatures, greedy and invalid ones included, in one call.
"""

import numpy as np
import pytest
import torch
from scipy.special import softmax as sp_softmax

import oracle
import oracle_pins as pins
import parity
from speculative_decoding_verification_82_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    binding.library()


def _show(name, st):
    print(f"\n[{name}] {st}")


def _random_parents(rng, N1):
    par = np.full(N1, -1, np.int32)
    for i in range(1, N1):
        par[i] = rng.integers(max(0, i - 4), i)  # bushy and deep enough
    return par


def test_walk_invariance_on_gpu():
    """The emitted token after each prefix follows that prefix's target row (chi-squared), and
    the walk matches the oracle on every unflagged trial."""
    ti = synth.tree_sample_tiny(seed=7, trials=100_000)
    g = parity.run_gpu_walk(ti)
    st = parity.compare_walk(g, parity.run_oracle_walk(ti, threads=16), ti)
    _show("walk V=8 1e5", st)
    T = float(ti.temperature)
    out, L = g["out_tokens"], g["accept_len"]
    p0 = sp_softmax(ti.meta["t0"].astype(np.float64) / T)
    p1 = sp_softmax(ti.meta["t1"].astype(np.float64) / T, axis=-1)
    assert pins.chi2_pvalue(np.bincount(out[:, 0], minlength=ti.V).astype(float), p0) > 1e-4
    for a in range(ti.V):
        sel = (L >= 1) & (out[:, 0] == a)
        if sel.sum() >= 400:
            assert pins.chi2_pvalue(np.bincount(out[sel, 1], minlength=ti.V).astype(float), p1[a]) > 1e-4


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("V", [1, 7, 33, 4096, 4097, 16385, 40000, 131072, 131075, 200000])
def test_walk_random_trees(dtype, V):
    rng = np.random.default_rng(V * 7 + len(dtype))
    N1 = int(rng.integers(2, 14))
    ti = synth.tree_sample(seed=V % 1000, B=6, V=V, temperature=1.0, dtype=dtype,
                           parents=_random_parents(rng, N1), draft_sigma=1.0)
    st = parity.compare_walk(parity.run_gpu_walk(ti), parity.run_oracle_walk(ti), ti)
    st0 = parity.compare_walk(parity.run_gpu_walk(ti, 0.0), parity.run_oracle_walk(ti, 0.0), ti)
    _show(f"walk {dtype} V={V} N1={N1}", (st, st0))


@pytest.mark.parametrize("seed", [0, 1])
def test_walk_benchmark_tree(seed):
    """B = 16, the 61-node EAGLE-2-like tree, V = 128256 bf16, T = 1: every request."""
    ti = synth.tree_sample(seed=seed)
    g = parity.run_gpu_walk(ti)
    st = parity.compare_walk(g, parity.run_oracle_walk(ti, threads=16), ti)
    _show(f"walk benchmark tree seed={seed}", st)
    assert st["errors"] == 0


def test_greedy_walk_equals_streaming_greedy_tree():
    """T = 0 on the greedy tree workload: the walk, the oracle and spec_verify_tree_greedy agree."""
    for pb in (0.0, 40.0):
        ti = synth.tree_greedy(seed=1, path_boost=pb)
        g = parity.run_gpu_walk(ti, 0.0)
        parity.compare_walk(g, parity.run_oracle_walk(ti, 0.0, threads=16), ti)
        s = parity.run_gpu_tree(ti)
        assert np.array_equal(g["accept_len"], s["accept_len"])
        assert np.array_equal(g["path_nodes"], s["path_nodes"])
        assert np.array_equal(g["out_tokens"], s["out_tokens"])


def test_walk_more_requests_than_clusters():
    rng = np.random.default_rng(3)
    ti = synth.tree_sample(seed=3, B=200, V=40000, parents=_random_parents(rng, 6), draft_sigma=1.0)
    st = parity.compare_walk(parity.run_gpu_walk(ti), parity.run_oracle_walk(ti, threads=16), ti)
    _show("walk B=200 V=40000", st)
    tiny = synth.tree_sample_tiny(seed=4, trials=3000)
    parity.compare_walk(parity.run_gpu_walk(tiny), parity.run_oracle_walk(tiny), tiny)


@pytest.mark.parametrize("B,V,dtype", [(40, 128256, "bf16"), (20, 131075, "f32"), (20, 147456, "f16")])
def test_walk_single_wave_geometry(B, V, dtype):
    """Batches that need more waves of 8-CTA clusters than of 6-CTA clusters: the stochastic walk
    takes the 6-CTA clusters that keep q in shared memory, and the greedy walk the 6-CTA
    instantiation without q (several requests per cluster at B = 40; a ragged vocabulary; the
    largest vocabulary 6 CTAs cover)."""
    rng = np.random.default_rng(B + V)
    ti = synth.tree_sample(seed=V % 97, B=B, V=V, dtype=dtype, parents=_random_parents(rng, 7), draft_sigma=1.0)
    st = parity.compare_walk(parity.run_gpu_walk(ti), parity.run_oracle_walk(ti, threads=16), ti)
    st0 = parity.compare_walk(parity.run_gpu_walk(ti, 0.0), parity.run_oracle_walk(ti, 0.0, threads=16), ti)
    _show(f"walk single wave B={B} V={V} {dtype}", (st, st0))
    assert st["errors"] == 0 and st0["errors"] == 0


def test_walk_limits():
    """The largest walk shapes: a tree of SPEC_MAX_WALK_NODES nodes (two interleaved chains)
    whose draft rows nearly equal its target rows, so that the stochastic walk descends over a
    hundred levels, and the greedy walk on it; then the largest vocabulary, SPEC_MAX_WALK_VOCAB
    (16-CTA clusters, no ragged tail)."""
    rng = np.random.default_rng(17)
    N1 = binding.MAX_WALK_NODES
    par = np.array([-1, 0] + [i - 2 for i in range(2, N1)], np.int32)  # two interleaved chains
    ti = synth.tree_sample(seed=17, B=2, V=3000, temperature=1.0, dtype="bf16", parents=par,
                           draft_sigma=0.05)
    o = parity.run_oracle_walk(ti)
    assert o["accept_len"].max() >= 100
    st = parity.compare_walk(parity.run_gpu_walk(ti), o, ti)
    st0 = parity.compare_walk(parity.run_gpu_walk(ti, 0.0), parity.run_oracle_walk(ti, 0.0), ti)
    _show(f"walk of {N1} nodes", (st, st0))
    ti = synth.tree_sample(seed=18, B=2, V=binding.MAX_WALK_VOCAB, temperature=1.0, dtype="f16",
                           parents=_random_parents(rng, 6), draft_sigma=1.0)
    st = parity.compare_walk(parity.run_gpu_walk(ti), parity.run_oracle_walk(ti), ti)
    st0 = parity.compare_walk(parity.run_gpu_walk(ti, 0.0), parity.run_oracle_walk(ti, 0.0), ti)
    _show(f"walk V={ti.V}", (st, st0))


@pytest.mark.parametrize("T", [0.05, 0.3, 2.5, 8.0])
def test_walk_temperatures(T):
    rng = np.random.default_rng(int(T * 100))
    ti = synth.tree_sample(seed=11, B=8, V=32000, temperature=T, parents=_random_parents(rng, 10))
    st = parity.compare_walk(parity.run_gpu_walk(ti), parity.run_oracle_walk(ti), ti)
    _show(f"walk T={T}", st)


def test_walk_edge_cases():
    V = 5000
    par = np.array([-1, 0, 0, 1, 1, 2], np.int32)
    base = synth.tree_sample(seed=21, B=8, V=V, dtype="f32", parents=par, draft_sigma=0.5)
    ti = base
    tgt, dft = ti.target.copy(), ti.draft.copy()
    tok, pa = ti.node_tokens.copy(), ti.parents.copy()
    pa[1, 3] = 4                      # parent not below the node
    tok[2, 4] = V + 5                 # token outside [0, V)
    pa[3, 0] = 0                      # root with a parent
    tgt[4, 0, 17] = np.nan            # NaN in the root row: always visited
    tgt[5, 0, :] = -np.inf            # all -inf root row
    dft[6, 0, 3] = np.inf             # +inf in the root's draft row
    dft[7, 3:] = np.nan               # draft rows of leaves: never read
    tgt[0, 5, 9] = np.nan             # node 5 is reachable only through node 2 of request 0
    ti = synth.TreeInputs("edge", "f32", 8, 5, V, tgt, tok, pa, draft=dft, r=ti.r, u=ti.u,
                          temperature=ti.temperature)
    g = parity.run_gpu_walk(ti)
    o = parity.run_oracle_walk(ti)
    parity.compare_walk(g, o, ti)
    assert list(o["err"][1:8]) == [oracle.ERR_BAD_TREE, oracle.ERR_BAD_TOKEN, oracle.ERR_BAD_TREE,
                                    oracle.ERR_NONFINITE, oracle.ERR_NONFINITE,
                                    oracle.ERR_NONFINITE, 0]
    g0 = parity.run_gpu_walk(ti, 0.0)
    parity.compare_walk(g0, parity.run_oracle_walk(ti, 0.0), ti)
    # the root alone: the token is drawn from the root row
    one = synth.tree_sample(seed=22, B=5, V=3000, parents=np.array([-1], np.int32))
    parity.compare_walk(parity.run_gpu_walk(one), parity.run_oracle_walk(one), one)
    parity.compare_walk(parity.run_gpu_walk(one, 0.0), parity.run_oracle_walk(one, 0.0), one)


def test_walk_masked_tokens():
    """-inf logits (masked tokens) in target and draft rows: q(x) = 0 accepts, p(x) = 0 rejects."""
    ti = synth.tree_sample(seed=31, B=8, V=9000, dtype="bf16",
                           parents=np.array([-1, 0, 0, 0, 1, 1], np.int32), draft_sigma=1.0)
    tgt = synth.decode(ti.target, "bf16").copy()
    dft = synth.decode(ti.draft, "bf16").copy()
    rng = np.random.default_rng(5)
    for b in range(ti.B):
        for n in range(6):
            tgt[b, n, rng.choice(ti.V, 500, replace=False)] = -np.inf
            dft[b, n, rng.choice(ti.V, 500, replace=False)] = -np.inf
        tgt[b, 0, ti.node_tokens[b, 1]] = -np.inf   # p(x) = 0 for child 1
        dft[b, 0, ti.node_tokens[b, 2]] = -np.inf   # q(x) = 0 for child 2
    ti2 = synth.TreeInputs("masked", "bf16", ti.B, ti.N, ti.V, synth.encode(tgt, "bf16"),
                           ti.node_tokens, ti.parents, draft=synth.encode(dft, "bf16"), r=ti.r,
                           u=ti.u, temperature=ti.temperature)
    g = parity.run_gpu_walk(ti2)
    st = parity.compare_walk(g, parity.run_oracle_walk(ti2), ti2)
    _show("walk masked", st)


def test_walk_repeatable_and_on_a_side_stream():
    ti = synth.tree_sample(seed=41, B=12, V=20000, parents=_random_parents(np.random.default_rng(1), 9))
    a = parity.run_gpu_walk(ti)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = parity.run_gpu_walk(ti)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_walk_per_request_temperatures():
    """Each request at its own temperature (greedy ones included) in one call, against the oracle
    with the same per-request temperatures; NaN and negative temperatures fail their request."""
    rng = np.random.default_rng(61)
    ti = synth.tree_sample(seed=61, B=14, V=32000, parents=_random_parents(rng, 12), draft_sigma=1.0)
    temps = np.array([0.0, 0.6, 1.0, 1.6, 0.05, 4.0, 0.0, 0.9, 1.2, 0.3, np.nan, -0.5, 0.7, 2.2],
                     np.float32)
    g = parity.run_gpu_walk(ti, 1.0, temperatures=temps)
    o = parity.run_oracle_walk(ti, 1.0, temperatures=temps)
    st = parity.compare_walk(g, o, ti)
    _show("walk per-request T", st)
    assert list(o["err"][10:12]) == [oracle.ERR_BAD_TEMP] * 2
    # a request's result equals a call at its own temperature
    one = parity.run_gpu_walk(ti, 1.6)
    assert np.array_equal(one["path_nodes"][3], g["path_nodes"][3])
    assert np.array_equal(one["out_tokens"][3], g["out_tokens"][3])
