"""GPU parity of prompt n-gram lookup drafting (spec_ngram_draft) against the CPU oracle, and the
drafted n-gram pipeline (lookup on the GPU, then spec_verify_ngram) on the n-gram workload."""

import numpy as np
import pytest
import torch

import oracle
import parity
from speculative_decoding_verification_82_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    binding.library()


def _gpu(ctx, lens, K, n_max=4, n_min=1):
    o = binding.spec_ngram_draft(parity.i32(ctx), parity.i32(lens), K, n_max=n_max, n_min=n_min)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in o.items()}


def _compare(g, o):
    assert np.array_equal(g["err_flags"], o["err"])
    assert np.array_equal(g["draft_tokens"], o["draft"]), np.argwhere(g["draft_tokens"] != o["draft"])[:5]
    assert np.array_equal(g["draft_len"], o["draft_len"])
    assert np.array_equal(g["match_n"], o["match_n"])
    assert np.array_equal(g["match_end"], o["match_end"])


@pytest.mark.parametrize("K,n_max,n_min", [(5, 4, 1), (1, 4, 1), (16, 8, 2), (5, 1, 1), (7, 32, 3),
                                         (256, 32, 1)])  # the largest K and n_max
def test_random_contexts(K, n_max, n_min):
    rng = np.random.default_rng(K * 100 + n_max)
    B, Lmax = 600, 300
    ctx = np.empty((B, Lmax), np.int32)
    for b in range(B):  # alphabets from 2 to 60 tokens: matches of every length occur
        ctx[b] = rng.integers(0, int(rng.integers(2, 61)), Lmax)
    lens = rng.integers(0, Lmax + 1, B).astype(np.int32)
    lens[:4] = [0, 1, 2, Lmax]
    g = _gpu(ctx, lens, K, n_max, n_min)
    o = oracle.ngram_draft_batch(ctx, lens, K, n_max, n_min, threads=8)
    _compare(g, o)
    assert (o["match_n"] > 0).sum() >= 20  # matches of several lengths occur


def test_invalid_lengths_and_long_contexts():
    rng = np.random.default_rng(9)
    B, Lmax = 6, 100_000
    ctx = rng.integers(0, 3000, (B, Lmax)).astype(np.int32)
    lens = np.array([Lmax, 77_777, -1, Lmax + 1, 0, 50_001], np.int32)
    ctx[5, 50_001 - 4: 50_001] = ctx[5, 1234: 1238]  # a planted 4-gram repeat
    g = _gpu(ctx, lens, 5)
    o = oracle.ngram_draft_batch(ctx, lens, 5)
    _compare(g, o)
    assert list(o["err"][2:4]) == [oracle.ERR_BAD_TOKEN] * 2
    assert o["match_n"][5] == 4 and o["match_end"][5] == 1238


def test_workload_contexts_give_the_workload_drafts():
    ctx, lens = synth.ngram_contexts(seed=2)
    g = _gpu(ctx, lens, 5)
    _compare(g, oracle.ngram_draft_batch(ctx, lens, 5, threads=8))
    assert np.array_equal(g["draft_tokens"], synth.ngram(seed=2).draft_tokens)


def test_drafted_pipeline_equals_verification_of_the_workload_drafts():
    """Lookup on the GPU feeding spec_verify_ngram gives what verifying the workload's own drafts
    gives (B = 256, V = 151936 bf16, T = 0.8), and the oracle agrees on the verification."""
    ctx, lens = synth.ngram_contexts(seed=0)
    ci = synth.ngram(seed=0)
    d = binding.spec_ngram_draft(parity.i32(ctx), parity.i32(lens), ci.K)
    tl = parity.to_device(ci.target, ci.dtype)
    r, u = parity.f32(ci.r), parity.f32(ci.u)
    a = binding.spec_verify_ngram(tl, d["draft_tokens"], r, u, float(ci.temperature))
    b = binding.spec_verify_ngram(tl, parity.i32(ci.draft_tokens), r, u, float(ci.temperature))
    torch.cuda.synchronize()
    for k in ("num_accepted", "out_tokens", "err_flags"):
        assert torch.equal(a[k], b[k]), k
    g = {k: v.cpu().numpy() for k, v in a.items()}
    g["accept_prob"] = np.zeros((ci.B, ci.K))  # not requested here
    o = parity.run_oracle_chain(ci, ngram=True, threads=16)
    ok = ((o["req_flag"] & (oracle.FLAG_ACCEPT_TIE | oracle.FLAG_CDF_TIE)) == 0) & (o["err"] == 0)
    assert np.array_equal(g["num_accepted"][ok], o["num_accepted"][ok])
    assert np.array_equal(g["out_tokens"][ok], o["out_tokens"][ok])
