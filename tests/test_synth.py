"""The seeded input generators: determinism, prefix property, ranges and workload structure."""

import numpy as np

from speculative_decoding_verification_82_gb300 import synth


def test_uniform_ranges_exact_fp32():
    r = synth.uniform_r(3, (1000, 7))
    u = synth.uniform_u(3, (5000,))
    assert r.dtype == np.float32 and u.dtype == np.float32
    assert (r > 0).all() and (r <= 1).all() and (u >= 0).all() and (u < 1).all()
    assert np.array_equal(r * np.float32(1 << 24), np.round(r * np.float32(1 << 24)))
    assert np.array_equal(u * np.float32(1 << 24), np.round(u * np.float32(1 << 24)))


def test_bf16_rounding_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -3.0, 1e-3], np.float32)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: rounds to even (1.0)
    h = synth.to_bf16_bits(x)
    back = synth.bf16_bits_to_f32(h)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == np.float32(1.015625)
    assert back[3] == -3.0 and abs(back[4] - 1e-3) < 1e-5


def test_deterministic_and_prefix():
    a = synth.chain_batched(seed=1, B=3, V=512)
    b = synth.chain_batched(seed=1, B=3, V=512)
    c = synth.chain_batched(seed=1, B=2, V=512)
    assert np.array_equal(a.target, b.target) and np.array_equal(a.draft_tokens, b.draft_tokens)
    assert np.array_equal(a.target[:2], c.target) and np.array_equal(a.draft[:2], c.draft)
    assert np.array_equal(a.r[:2], c.r) and np.array_equal(a.u[:2], c.u)
    d = synth.chain_batched(seed=2, B=3, V=512)
    assert not np.array_equal(a.target, d.target)


def test_chain_batched_spikes():
    ci = synth.chain_batched(seed=0, B=2, K=2, V=4096)
    boosts = synth.zipf_boosts()
    assert abs(boosts[0] - 10) < 1e-6 and abs(boosts[-1] - 2) < 1e-6
    assert (np.diff(boosts) < 0).all()
    assert ci.target.shape == (2, 3, 4096) and ci.draft.shape == (2, 2, 4096)
    assert ci.draft_tokens.min() >= 0 and ci.draft_tokens.max() < 4096


def test_tree_shape():
    par = synth.eagle_tree_parents()
    assert par.size == 61 and par[0] == -1
    assert all(0 <= par[i] < i for i in range(1, 61))
    depth = np.zeros(61, int)
    for i in range(1, 61):
        depth[i] = depth[par[i]] + 1
    assert depth.max() == 6
    assert [int((depth == d).sum()) for d in range(1, 7)] == [10, 16, 12, 10, 6, 6]
    assert int((par == 0).sum()) == 10  # top-10 at the root
    ti = synth.tree_greedy(seed=0, B=2, V=1000)
    for b in range(2):
        for p in range(61):
            kids = np.nonzero(par == p)[0]
            toks = ti.node_tokens[b, kids]
            assert len(set(toks.tolist())) == len(toks)  # distinct siblings


def test_ngram_drafts_are_prompt_continuations():
    ng = synth.ngram(seed=0, B=8, V=1000)
    prompt, starts = ng.meta["prompt"], ng.meta["starts"]
    for b in range(8):
        s = starts[b]
        assert np.array_equal(ng.draft_tokens[b], prompt[s + 4: s + 4 + ng.K])
    assert ng.draft is None and ng.target.dtype == np.uint16
