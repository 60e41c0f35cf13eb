"""The parity checker's flagged-tie rule has power: on the CPU, with the oracle's own outputs in
the place of a GPU result, it accepts the oracle's outcome and the admissible alternatives of a
flagged tie (the other side of a CDF boundary that u sits on, the other decision of an accept test
that r sits on), and rejects planted wrong answers (a token one interval further, a zero-weight
token, an accepted length that no decision gives, a walk path that neither decision gives).

Ties are made on purpose: u is moved onto a boundary of the oracle's own CDF of a draw, r onto the
oracle's own alpha, both rounded to the grid of 2^-24 the uniforms live on.
"""

import numpy as np
import pytest

import oracle

pytest.importorskip("torch")
import parity  # noqa: E402
from speculative_decoding_verification_82_gb300 import synth  # noqa: E402

U24 = float(1 << 24)


def _chain_case(seed=3, B=6, K=3, V=1500):
    rng = np.random.default_rng(seed)
    t = rng.normal(0, 2.0, (B, K + 1, V)).astype(np.float32)
    d = (t[:, :K] + rng.normal(0, 1.0, (B, K, V))).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    r = ((rng.integers(0, 1 << 24, (B, K)) + 1) / U24).astype(np.float32)
    u = (rng.integers(0, 1 << 24, B) / U24).astype(np.float32)
    return synth.ChainInputs("checker", "f32", B, K, V, np.float32(1.0), t, d, x, r, u)


def _as_gpu(o, K):
    """The oracle's chain outputs in the layout of the GPU result."""
    n = o["num_accepted"]
    return dict(num_accepted=n.copy(), out_tokens=o["out_tokens"].copy(),
                residual_mass=o["mass"][np.arange(n.size), np.minimum(n, K)].astype(np.float32),
                err_flags=o["err"].copy(), accept_prob=o["alpha"].astype(np.float32),
                cand_tokens=o["cand"].copy(), pos_mass=o["mass"].astype(np.float32))


def _positive(w, lo, hi):
    return [i for i in range(lo, hi) if w[i] > 0]


@pytest.mark.parametrize("ngram", [False, True])
def test_chain_flagged_draw(ngram):
    ci = _chain_case()
    o = parity.run_oracle_chain(ci, ngram=ngram)
    b = 0
    n = int(o["num_accepted"][b])
    d = oracle.chain_draw_rows(ci.dtype, ci.target, ci.draft, ci.B, ci.K, ci.V,
                               float(ci.temperature), ci.draft_tokens, b, ngram=ngram)
    w, cdf = d["w"], d["cdf"]
    assert d["err"] == 0
    pos = _positive(w[n], 0, ci.V)
    t = pos[len(pos) // 2]  # a boundary in the middle of the CDF: u onto cdf[t]
    ci.u[b] = np.float32(round(cdf[n][t] * U24) / U24)
    o = parity.run_oracle_chain(ci, ngram=ngram)
    assert o["num_accepted"][b] == n and o["pos_flag"][b][n] & oracle.FLAG_CDF_TIE
    g = _as_gpu(o, ci.K)
    st = parity.check_chain(g, o, ci)
    assert not st["failures"] and st["flagged_strict"] >= 1
    pick = int(o["out_tokens"][b][n])
    # the token on the other side of the boundary is admissible
    other = pos[pos.index(t) + 1] if pick == t else t
    g2 = _as_gpu(o, ci.K)
    g2["out_tokens"][b][n] = other
    g2["cand_tokens"][b][n] = other
    st = parity.check_chain(g2, o, ci)
    assert not st["failures"], st["failures"]
    assert st["admissible_deviations"] == 1
    # a later token whose interval starts more than the band above u is not
    band = parity._tie_band(float(o["mass"][b][n]), widened=(not ngram and n < ci.K))
    far = next(i for i in pos if i > max(pick, other) and cdf[n][i - 1] - float(ci.u[b]) > 2 * band)
    g3 = _as_gpu(o, ci.K)
    g3["out_tokens"][b][n] = far
    assert parity.check_chain(g3, o, ci)["failures"]
    # a zero-weight token is never admissible, wherever its (empty) interval lies (unless its largest
    # weight within fp32 precision is positive and the draw is in the widened tier)
    zeros = [i for i in range(ci.V) if d["wmax"][n][i] == 0]
    if zeros:
        z = min(zeros, key=lambda i: abs(cdf[n][i] - float(ci.u[b])))
        g4 = _as_gpu(o, ci.K)
        g4["out_tokens"][b][n] = z
        assert parity.check_chain(g4, o, ci)["failures"]
    # an unflagged request admits only the oracle's token
    b2 = next(i for i in range(1, ci.B) if not o["req_flag"][i])
    n2 = int(o["num_accepted"][b2])
    g5 = _as_gpu(o, ci.K)
    g5["out_tokens"][b2][n2] = (int(o["out_tokens"][b2][n2]) + 1) % ci.V
    assert parity.check_chain(g5, o, ci)["failures"]


def test_chain_flagged_accept_test():
    ci = _chain_case(seed=5)
    o = parity.run_oracle_chain(ci)
    b, k = 1, 0
    a = float(o["alpha"][b][k])
    assert 0.01 < a < 0.99
    ci.r[b][k] = np.float32(a)  # r on alpha: either decision is admissible
    o = parity.run_oracle_chain(ci)
    assert o["req_flag"][b] & oracle.FLAG_ACCEPT_TIE
    assert not parity.check_chain(_as_gpu(o, ci.K), o, ci)["failures"]
    # the other decision, as the oracle gives it with r moved off alpha to the other side
    alt = synth.ChainInputs(**{**ci.__dict__, "r": ci.r.copy()})
    accepted = float(ci.r[b][k]) <= a
    alt.r[b][k] = np.float32(a + 1e-3) if accepted else np.float32(a - 1e-3)
    oa = parity.run_oracle_chain(alt)
    assert oa["num_accepted"][b] != o["num_accepted"][b]
    g = _as_gpu(o, ci.K)
    g["num_accepted"][b] = oa["num_accepted"][b]
    g["out_tokens"][b] = oa["out_tokens"][b]
    g["residual_mass"][b] = oa["mass"][b][min(int(oa["num_accepted"][b]), ci.K)]
    st = parity.check_chain(g, o, ci)
    assert not st["failures"], st["failures"]
    # an accepted length that no decision gives (a rejection at an unflagged position moved)
    b2 = next(i for i in range(ci.B) if i != b and not o["req_flag"][i] and o["num_accepted"][i] < ci.K)
    g2 = _as_gpu(o, ci.K)
    g2["num_accepted"][b2] += 1
    n2 = int(g2["num_accepted"][b2])
    g2["out_tokens"][b2][: n2] = ci.draft_tokens[b2][: n2]
    g2["out_tokens"][b2][n2] = o["cand"][b2][min(n2, ci.K)]
    assert parity.check_chain(g2, o, ci)["failures"]


def _walk_case(seed=7, V=600):
    ti = synth.tree_sample(seed=seed, B=4, V=V, dtype="f32")
    return ti


def _walk_gpu(o, b=None, alt=None):
    g = dict(accept_len=o["accept_len"].copy(), path_nodes=o["path"].copy(),
             out_tokens=o["out_tokens"].copy(), residual_mass=o["mass"].astype(np.float32),
             err_flags=o["err"].copy(), accept_prob=o["alpha"].astype(np.float32))
    if alt is not None:
        g["accept_len"][b] = alt["accept_len"]
        g["path_nodes"][b] = alt["path"]
        g["out_tokens"][b] = alt["out_tokens"]
        g["residual_mass"][b] = alt["mass"]
        g["accept_prob"][b] = alt["alpha"]
    return g


def test_walk_flagged_accept_test_and_draw():
    ti = _walk_case()
    o = parity.run_oracle_walk(ti)
    # an accept tie on the first tested child of request 0
    b = 0
    c = int(np.nonzero(o["alpha"][b] >= 0)[0][0])
    a = float(o["alpha"][b][c])
    if not 0.01 < a < 0.99:
        pytest.skip("the seeded tree's first test is decided far from a tie")
    ti.r[b][c] = np.float32(a)
    o = parity.run_oracle_walk(ti)
    assert o["req_flag"][b] & oracle.FLAG_ACCEPT_TIE
    assert not parity.check_walk(_walk_gpu(o), o, ti)["failures"]
    alt = oracle.tree_sample_alt(ti.dtype, ti.target, ti.draft, ti.B, ti.N, ti.V, float(ti.temperature),
                                 ti.node_tokens, ti.parents, ti.r, ti.u, b, True)
    assert alt["accept_len"] != o["accept_len"][b] or not np.array_equal(alt["path"], o["path"][b])
    st = parity.check_walk(_walk_gpu(o, b, alt), o, ti)
    assert not st["failures"] and st["flipped_accept_ties"] == 1, st["failures"]
    # a path that neither decision gives
    g = _walk_gpu(o)
    b2 = next(i for i in range(1, ti.B) if not o["req_flag"][i])
    kids = np.nonzero(ti.parents[b2] == 0)[0]
    wrong = int(kids[-1]) if o["path"][b2][1] != kids[-1] else int(kids[0])
    g["accept_len"][b2] = 1
    g["path_nodes"][b2][:] = -1
    g["path_nodes"][b2][:2] = [0, wrong]
    assert parity.check_walk(g, o, ti)["failures"]
    # a flagged draw: u onto a boundary of request b2's final draw
    d = oracle.tree_sample_alt(ti.dtype, ti.target, ti.draft, ti.B, ti.N, ti.V, float(ti.temperature),
                               ti.node_tokens, ti.parents, ti.r, ti.u, b2, False)
    pos = _positive(d["draw_w"], 0, ti.V)
    t = pos[len(pos) // 2]
    ti.u[b2] = np.float32(round(d["draw_cdf"][t] * U24) / U24)
    o = parity.run_oracle_walk(ti)
    assert o["req_flag"][b2] & (oracle.FLAG_CDF_TIE | oracle.FLAG_CDF_TIE_WIDE)
    L = int(o["accept_len"][b2])
    pick = int(o["out_tokens"][b2][L])
    other = pos[pos.index(t) + 1] if pick == t else t
    g = _walk_gpu(o)
    g["out_tokens"][b2][L] = other
    st = parity.check_walk(g, o, ti)
    assert not st["failures"] and st["admissible_deviations"] == 1, st["failures"]
    band = parity._tie_band(float(o["mass"][b2]), True)
    u2 = float(ti.u[b2])
    g["out_tokens"][b2][L] = next(i for i in pos if i > max(pick, other) and d["draw_cdf"][i - 1] - u2 > 2 * band)
    assert parity.check_walk(g, o, ti)["failures"]
