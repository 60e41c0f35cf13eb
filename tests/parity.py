"""Helpers for the GPU-vs-oracle parity tests: move seeded inputs to the device, run the CUDA
path through the C ABI (via the binding), run the oracle on the same host arrays, compare.

The comparison rules follow the parity contract:
  * error bits, greedy results and tree results: bit-exact;
  * accepted lengths and emitted tokens: bit-exact unless the oracle puts the request in the
    flagged-tie set (|r - alpha| within 1e-6, or a CDF crossing within the tie band of u);
    flagged requests must still produce one of the valid outcomes;
  * per-position candidates: bit-exact unless that position's CDF crossing is flagged;
  * probabilities (alpha, residual masses, optional p / q rows): within 1e-5 absolute.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from speculative_decoding_verification_82_gb300 import binding

PROB_TOL = 1e-5
TIE_TOL = oracle.DEFAULT_TOL


def to_device(storage: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    a = np.ascontiguousarray(storage)
    if dtype == "bf16":
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    elif dtype == "f16":
        t = torch.from_numpy(a.view(np.float16))
    else:
        t = torch.from_numpy(a.astype(np.float32, copy=False))
    return t.to(device)


def i32(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def f32(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def run_gpu_chain(ci, ngram: bool = False, probs: bool = False, workspace=None, diag: bool = True) -> dict:
    dev = "cuda"
    B, K, V = ci.B, ci.K, ci.V
    tl = to_device(ci.target, ci.dtype)
    dl = None if (ngram or ci.draft is None) else to_device(ci.draft, ci.dtype)
    x, r, u = i32(ci.draft_tokens), f32(ci.r), f32(ci.u)
    ap = torch.full((B, K), -1.0, device=dev)
    ct = torch.full((B, K + 1), -7, dtype=torch.int32, device=dev) if diag else None
    pm = torch.full((B, K + 1), -1.0, device=dev) if diag else None
    tp = torch.zeros((B, K + 1, V), device=dev) if probs else None
    dp = torch.zeros((B, K, V), device=dev) if (probs and not ngram) else None
    if ngram:
        o = binding.spec_verify_ngram(tl, x, r, u, float(ci.temperature), workspace=workspace,
                                      accept_prob=ap, cand_tokens=ct, pos_mass=pm, target_probs=tp)
    else:
        o = binding.spec_verify_chain(tl, dl, x, r, u, float(ci.temperature), workspace=workspace,
                                      accept_prob=ap, cand_tokens=ct, pos_mass=pm, target_probs=tp,
                                      draft_probs=dp)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in o.items()}
    res["accept_prob"] = ap.cpu().numpy()
    if diag:
        res.update(cand_tokens=ct.cpu().numpy(), pos_mass=pm.cpu().numpy())
    if probs:
        res["target_probs"] = tp.cpu().numpy()
        if dp is not None:
            res["draft_probs"] = dp.cpu().numpy()
    return res


def run_oracle_chain(ci, ngram: bool = False, threads: int = 8, requests=None) -> dict:
    if ngram:
        return oracle.verify_ngram(ci.dtype, ci.target, ci.B, ci.K, ci.V, float(ci.temperature),
                                   ci.draft_tokens, ci.r, ci.u, threads=threads, requests=requests)
    return oracle.verify_chain(ci.dtype, ci.target, ci.draft, ci.B, ci.K, ci.V,
                               float(ci.temperature), ci.draft_tokens, ci.r, ci.u, threads=threads,
                               requests=requests)


def compare_chain(g: dict, o: dict, ci, requests=None) -> dict:
    """Asserts parity of a chain / n-gram call; returns counts (flagged-tie set size etc.)."""
    idx = np.arange(ci.B) if requests is None else np.arange(*requests)
    K = ci.K
    greedy = float(ci.temperature) == 0.0
    err_o, err_g = o["err"][idx], g["err_flags"][idx]
    assert np.array_equal(err_o, err_g), ("error bits differ", np.nonzero(err_o != err_g)[0][:10])
    ok = err_o == 0
    bad = idx[~ok]
    assert (g["num_accepted"][bad] == 0).all() and (g["out_tokens"][bad] == -1).all()
    good = idx[ok]
    if K:
        da = np.abs(g["accept_prob"][good] - o["alpha"][good])
        assert da.size == 0 or da.max() <= (0 if greedy else PROB_TOL), ("alpha", da.max())
    cdf_flag = (o["pos_flag"][good] & oracle.FLAG_CDF_TIE) != 0
    if "pos_mass" in g:
        dm = np.abs(g["pos_mass"][good] - o["mass"][good])
        assert dm.size == 0 or dm.max() <= PROB_TOL, ("position mass", dm.max())
        cm = (g["cand_tokens"][good] != o["cand"][good]) & ~cdf_flag
        assert not cm.any(), ("candidate tokens differ", np.argwhere(cm)[:10])
    flagged = (o["req_flag"][good] & (oracle.FLAG_ACCEPT_TIE | oracle.FLAG_CDF_TIE)) != 0
    ex = good[~flagged]
    assert np.array_equal(g["num_accepted"][ex], o["num_accepted"][ex]), "accepted lengths differ"
    assert np.array_equal(g["out_tokens"][ex], o["out_tokens"][ex]), "emitted tokens differ"
    n_g = g["num_accepted"][good]
    dmass = np.abs(g["residual_mass"][good] - o["mass"][good, n_g])
    assert dmass.size == 0 or dmass.max() <= PROB_TOL, ("residual mass", dmass.max())
    for b in good[flagged]:  # flagged ties: any valid outcome
        n = int(g["num_accepted"][b])
        a, r = o["alpha"][b], ci.r[b]
        assert all(r[k] <= a[k] + TIE_TOL for k in range(n))
        assert n == K or r[n] > a[n] - TIE_TOL
        out = g["out_tokens"][b]
        assert list(out[:n]) == list(ci.draft_tokens[b][:n])
        assert 0 <= out[n] < ci.V
        assert (out[n + 1:] == -1).all()
    return dict(requests=int(idx.size), errors=int((~ok).sum()), flagged=int(flagged.sum()),
                cdf_flagged_positions=int(cdf_flag.sum()),
                mean_accepted=float(n_g.mean()) if n_g.size else 0.0)


def run_gpu_tree(ti, workspace=None) -> dict:
    tl = to_device(ti.target, ti.dtype)
    am = torch.full((ti.B, ti.N + 1), -7, dtype=torch.int32, device="cuda")
    o = binding.spec_verify_tree_greedy(tl, i32(ti.node_tokens), i32(ti.parents),
                                        workspace=workspace, node_argmax=am)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in o.items()}
    res["node_argmax"] = am.cpu().numpy()
    return res


def run_oracle_tree(ti, threads: int = 8) -> dict:
    return oracle.verify_tree_greedy(ti.dtype, ti.target, ti.B, ti.N, ti.V, ti.node_tokens,
                                     ti.parents, threads=threads)


def compare_tree(g: dict, o: dict) -> dict:
    assert np.array_equal(g["err_flags"], o["err"]), "tree error bits differ"
    ok = o["err"] == 0
    assert np.array_equal(g["node_argmax"][ok], o["amax"][ok]), "row argmax differs"
    assert np.array_equal(g["accept_len"], o["accept_len"]), "accepted lengths differ"
    assert np.array_equal(g["path_nodes"], o["path"]), "paths differ"
    assert np.array_equal(g["out_tokens"], o["out_tokens"]), "emitted tokens differ"
    return dict(requests=int(ok.size), mean_accepted=float(o["accept_len"].mean()))


# ------------------------------------------------------------------------ tree walk ----
def run_gpu_walk(ti, temperature=None, temperatures=None) -> dict:
    T = float(ti.temperature if temperature is None else temperature)
    sampled = T > 0 or temperatures is not None
    tl = to_device(ti.target, ti.dtype)
    dl = to_device(ti.draft, ti.dtype) if (sampled and ti.draft is not None) else None
    r = f32(ti.r) if sampled else None
    u = f32(ti.u) if sampled else None
    tt = f32(temperatures) if temperatures is not None else None
    ap = torch.full((ti.B, ti.N + 1), -7.0, device="cuda")
    o = binding.spec_verify_tree_walk(tl, dl, i32(ti.node_tokens), i32(ti.parents), r, u, T,
                                      accept_prob=ap, temperatures=tt)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in o.items()}
    res["accept_prob"] = ap.cpu().numpy()
    return res


def run_oracle_walk(ti, temperature=None, threads: int = 8, temperatures=None) -> dict:
    T = float(ti.temperature if temperature is None else temperature)
    sampled = T > 0 or temperatures is not None
    return oracle.verify_tree_sample(ti.dtype, ti.target, ti.draft if sampled else None, ti.B, ti.N,
                                     ti.V, T, ti.node_tokens, ti.parents,
                                     ti.r if sampled else None, ti.u if sampled else None,
                                     threads=threads, temperatures=temperatures)


def compare_walk(g: dict, o: dict, ti) -> dict:
    """Parity of a tree walk: error bits exact; unflagged requests exact (path, tokens, the set of
    children tested); alpha of the children tested and the residual mass within 1e-5; flagged
    requests end on a valid path."""
    assert np.array_equal(g["err_flags"], o["err"]), ("walk error bits differ",
                                                      np.nonzero(g["err_flags"] != o["err"])[0][:10])
    ok = o["err"] == 0
    bad = np.nonzero(~ok)[0]
    assert (g["accept_len"][bad] == 0).all() and (g["out_tokens"][bad] == -1).all()
    assert (g["path_nodes"][bad] == -1).all() and (g["accept_prob"][bad] == -1).all()
    flagged = (o["req_flag"] & (oracle.FLAG_ACCEPT_TIE | oracle.FLAG_CDF_TIE)) != 0
    ex = np.nonzero(ok & ~flagged)[0]
    assert np.array_equal(g["accept_len"][ex], o["accept_len"][ex]), "accepted lengths differ"
    assert np.array_equal(g["path_nodes"][ex], o["path"][ex]), "paths differ"
    assert np.array_equal(g["out_tokens"][ex], o["out_tokens"][ex]), "emitted tokens differ"
    tested_g, tested_o = g["accept_prob"][ex] >= 0, o["alpha"][ex] >= 0
    assert np.array_equal(tested_g, tested_o), "children tested differ"
    da = np.abs(g["accept_prob"][ex] - o["alpha"][ex])[tested_o]
    assert da.size == 0 or da.max() <= PROB_TOL, ("alpha", da.max())
    dm = np.abs(g["residual_mass"][ex] - o["mass"][ex])
    assert dm.size == 0 or dm.max() <= PROB_TOL, ("residual mass", dm.max())
    for b in np.nonzero(ok & flagged)[0]:  # any valid outcome
        L = int(g["accept_len"][b])
        path = g["path_nodes"][b]
        assert path[0] == 0 and (path[L + 1:] == -1).all()
        for j in range(1, L + 1):
            assert ti.parents[b][path[j]] == path[j - 1]
            assert g["out_tokens"][b][j - 1] == ti.node_tokens[b][path[j]]
        assert 0 <= g["out_tokens"][b][L] < ti.V and (g["out_tokens"][b][L + 1:] == -1).all()
    return dict(requests=int(ok.size), errors=int((~ok).sum()), flagged=int(flagged.sum()),
                mean_accepted=float(g["accept_len"][ok].mean()) if ok.any() else 0.0,
                max_alpha_diff=float(da.max()) if da.size else 0.0)
