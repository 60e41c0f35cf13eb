"""Helpers for the GPU-vs-oracle parity tests: move seeded inputs to the device, run the CUDA
path through the C ABI (via the binding), run the oracle on the same host arrays, compare.

The comparison rules follow the parity contract:
  * error bits, greedy results and tree results: bit-exact;
  * accepted lengths and emitted tokens: bit-exact, except in the flagged-tie set, which the
    oracle reports in two tiers (strict: |r - alpha| or a CDF crossing within 1e-6 of the uniform;
    widened: within 1e-6 / S of a residual of total S < 1, not within 1e-6).  There an accept test
    admits either decision (for a walk, the oracle's outcome with that test decided the other way
    must then match), and a draw admits a positive-weight token whose CDF interval comes within
    the band of u, as the oracle's weights and CDF of that draw decide;
  * per-position candidates: likewise;
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


def run_gpu_chain(ci, ngram: bool = False, probs: bool = False, workspace=None, diag: bool = True,
                  temperatures=None, hot: bool = False) -> dict:
    """One call through the binding.  diag: ask for the per-position outputs too; hot: ask for no
    optional output at all (the configuration the benchmark times), so alpha is not checked."""
    dev = "cuda"
    B, K, V = ci.B, ci.K, ci.V
    tl = to_device(ci.target, ci.dtype)
    dl = None if (ngram or ci.draft is None) else to_device(ci.draft, ci.dtype)
    x, r, u = i32(ci.draft_tokens), f32(ci.r), f32(ci.u)
    ap = None if hot else torch.full((B, K), -1.0, device=dev)
    ct = torch.full((B, K + 1), -7, dtype=torch.int32, device=dev) if diag else None
    pm = torch.full((B, K + 1), -1.0, device=dev) if diag else None
    tp = torch.zeros((B, K + 1, V), device=dev) if probs else None
    dp = torch.zeros((B, K, V), device=dev) if (probs and not ngram) else None
    tt = f32(temperatures) if temperatures is not None else None
    if ngram:
        o = binding.spec_verify_ngram(tl, x, r, u, float(ci.temperature), workspace=workspace,
                                      accept_prob=ap, cand_tokens=ct, pos_mass=pm, target_probs=tp,
                                      temperatures=tt)
    else:
        o = binding.spec_verify_chain(tl, dl, x, r, u, float(ci.temperature), workspace=workspace,
                                      accept_prob=ap, cand_tokens=ct, pos_mass=pm, target_probs=tp,
                                      draft_probs=dp, temperatures=tt)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in o.items()}
    if ap is not None:
        res["accept_prob"] = ap.cpu().numpy()
    if diag:
        res.update(cand_tokens=ct.cpu().numpy(), pos_mass=pm.cpu().numpy())
    if probs:
        res["target_probs"] = tp.cpu().numpy()
        if dp is not None:
            res["draft_probs"] = dp.cpu().numpy()
    return res


def run_oracle_chain(ci, ngram: bool = False, threads: int = 8, requests=None, temperatures=None) -> dict:
    if ngram:
        o = oracle.verify_ngram(ci.dtype, ci.target, ci.B, ci.K, ci.V, float(ci.temperature),
                                ci.draft_tokens, ci.r, ci.u, threads=threads, requests=requests,
                                temperatures=temperatures)
    else:
        o = oracle.verify_chain(ci.dtype, ci.target, ci.draft, ci.B, ci.K, ci.V,
                                float(ci.temperature), ci.draft_tokens, ci.r, ci.u, threads=threads,
                                requests=requests, temperatures=temperatures)
    o["ngram"] = ngram
    o["temperatures"] = None if temperatures is None else np.asarray(temperatures, np.float32)
    return o


def draw_admissible(w: np.ndarray, cdf: np.ndarray, u: float, t: int, band: float, wmax=None) -> bool:
    """Token t is an admissible outcome of a draw with weights w and normalised CDF cdf (the
    oracle's): it has positive weight (or, in the widened tier, a positive largest weight wmax
    within fp32 precision) and its interval [cdf[t-1], cdf[t]) of u comes within `band` of the
    uniform u that was used."""
    if not (0 <= t < w.size):
        return False
    if not (w[t] > 0 or (wmax is not None and wmax[t] > 0)):
        return False
    lo = cdf[t - 1] if t > 0 else 0.0
    return lo - band <= u <= cdf[t] + band


def _tie_band(mass: float, widened: bool) -> float:
    """The band of a flagged draw: 1e-6, or 1e-6 / S where reading R10 / R14 widens it (a residual
    of total S < 1)."""
    return TIE_TOL / mass if (widened and 0.0 < mass < 1.0) else TIE_TOL


def check_chain(g: dict, o: dict, ci, requests=None) -> dict:
    """Parity of a chain / n-gram call without asserting: returns counts and a list of failures.

    Error bits, alpha (1e-5) and residual masses (1e-5) must match.  A request's accepted length
    must follow the oracle's decisions, except that an accept test within 1e-6 of alpha admits
    either decision.  Its emitted token must be the oracle's candidate at that position, or, where
    the oracle flags the draw as a tie, a positive-weight token whose CDF interval comes within
    the tie band of u (the oracle's weights and CDF of that draw decide)."""
    idx = np.arange(ci.B) if requests is None else np.arange(*requests)
    K, V = ci.K, ci.V
    T = float(ci.temperature)
    temps = o.get("temperatures")  # per-request temperatures, when the call took them

    def temp(b):
        return T if temps is None else float(temps[b])

    greedy = T == 0.0 and temps is None
    ngram = bool(o.get("ngram", False))
    fails = []
    err_o, err_g = o["err"][idx], g["err_flags"][idx]
    if not np.array_equal(err_o, err_g):
        fails.append(("error bits differ", np.nonzero(err_o != err_g)[0][:10].tolist()))
    ok = err_o == 0
    bad = idx[~ok]
    if not ((g["num_accepted"][bad] == 0).all() and (g["out_tokens"][bad] == -1).all()):
        fails.append(("failed requests emit something", bad[:10].tolist()))
    good = idx[ok]
    if K and "accept_prob" in g:
        da = np.abs(g["accept_prob"][good] - o["alpha"][good])
        if da.size and da.max() > (0 if greedy else PROB_TOL):
            fails.append(("alpha", float(da.max())))
    cdf_flag = (o["pos_flag"][good] & (oracle.FLAG_CDF_TIE | oracle.FLAG_CDF_TIE_WIDE)) != 0
    if "pos_mass" in g:
        dm = np.abs(g["pos_mass"][good] - o["mass"][good])
        if dm.size and dm.max() > PROB_TOL:
            fails.append(("position mass", float(dm.max())))
    rf = o["req_flag"][good]
    strict = (rf & oracle.FLAGS_STRICT) != 0
    wide_only = ((rf & oracle.FLAGS_WIDE) != 0) & ~strict
    n_g = g["num_accepted"][good]
    dmass = np.abs(g["residual_mass"][good] - o["mass"][good, np.minimum(n_g, K)])
    if dmass.size and dmass.max() > PROB_TOL:
        fails.append(("residual mass", float(dmass.max())))
    rows = {}

    def draw_rows(b):
        if b not in rows:
            rows[b] = oracle.chain_draw_rows(ci.dtype, ci.target, ci.draft, ci.B, K, V, temp(b),
                                             ci.draft_tokens, int(b), ngram=ngram)
        return rows[b]

    def admissible(b, k, t):
        """Token t at position k of request b: the candidate, or an admissible tie outcome."""
        if t == o["cand"][b][k]:
            return True, False
        if temp(b) == 0.0 or not (o["pos_flag"][b][k] & (oracle.FLAG_CDF_TIE | oracle.FLAG_CDF_TIE_WIDE)):
            return False, False
        d = draw_rows(b)
        widened = (not ngram) and k < K
        band = _tie_band(float(o["mass"][b][k]), widened)
        wmax = d["wmax"][k] if (widened and o["pos_flag"][b][k] & oracle.FLAG_CDF_TIE_WIDE) else None
        return (d["err"] == 0 and draw_admissible(d["w"][k], d["cdf"][k], float(ci.u[b]), int(t), band,
                                                  wmax)), True

    deviations = 0
    cand_dev = 0
    if "cand_tokens" in g:
        for b in good:
            for k in range(K + 1):
                t = int(g["cand_tokens"][b][k])
                good_t, dev = admissible(b, k, t)
                if not good_t:
                    fails.append(("candidate token", int(b), k, t, int(o["cand"][b][k])))
                cand_dev += int(dev)
    for b in good:
        n = int(g["num_accepted"][b])
        out = g["out_tokens"][b]
        a, r = o["alpha"][b], ci.r[b]
        if temp(b) == 0.0:
            if n != o["num_accepted"][b] or not np.array_equal(out, o["out_tokens"][b]):
                fails.append(("greedy outcome differs", int(b)))
            continue

        def tie(k):
            return abs(float(r[k]) - float(a[k])) <= TIE_TOL

        if not (0 <= n <= K and all(float(r[k]) <= a[k] or tie(k) for k in range(n))
                and (n == K or float(r[n]) > a[n] or tie(n))):
            fails.append(("accepted length not admissible", int(b), n, int(o["num_accepted"][b])))
            continue
        if list(out[:n]) != list(ci.draft_tokens[b][:n]) or not (out[n + 1:] == -1).all():
            fails.append(("accepted prefix or padding differs", int(b)))
            continue
        good_t, dev = admissible(b, n, int(out[n]))
        if not good_t:
            fails.append(("emitted token not admissible", int(b), n, int(out[n]), int(o["cand"][b][n])))
        deviations += int(dev or n != o["num_accepted"][b])
    return dict(requests=int(idx.size), errors=int((~ok).sum()), flagged=int((strict | wide_only).sum()),
                flagged_strict=int(strict.sum()), flagged_wide_only=int(wide_only.sum()),
                admissible_deviations=deviations, cdf_flagged_positions=int(cdf_flag.sum()),
                candidate_deviations=cand_dev,
                mean_accepted=float(n_g.mean()) if n_g.size else 0.0, failures=fails)


def compare_chain(g: dict, o: dict, ci, requests=None) -> dict:
    """Asserts parity of a chain / n-gram call (see check_chain); returns the counts."""
    st = check_chain(g, o, ci, requests)
    assert not st["failures"], st["failures"][:10]
    return st


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
    o = oracle.verify_tree_sample(ti.dtype, ti.target, ti.draft if sampled else None, ti.B, ti.N,
                                  ti.V, T, ti.node_tokens, ti.parents,
                                  ti.r if sampled else None, ti.u if sampled else None,
                                  threads=threads, temperatures=temperatures)
    o["temperature"], o["temperatures"] = T, temperatures  # (the settings the walk was run with)
    return o


def check_walk(g: dict, o: dict, ti, temperature=None, temperatures=None) -> dict:
    """Parity of a tree walk without asserting: returns counts and a list of failures.

    Error bits must match.  A request whose path is the oracle's must emit the oracle's tokens,
    except that a draw the oracle flags as a tie admits a positive-weight token whose CDF interval
    comes within the tie band of u; the children it tested, their alpha (1e-5) and its residual
    mass (1e-5) must match.  A request whose path differs must be flagged for an accept tie and
    match the oracle's walk with the first flagged test decided the other way (same rules)."""
    if temperature is None:
        temperature = o.get("temperature", ti.temperature)
    if temperatures is None:
        temperatures = o.get("temperatures")
    T = float(temperature)
    sampled = T > 0 or temperatures is not None
    fails = []
    if not np.array_equal(g["err_flags"], o["err"]):
        fails.append(("walk error bits differ", np.nonzero(g["err_flags"] != o["err"])[0][:10].tolist()))
    ok = o["err"] == 0
    bad = np.nonzero(~ok)[0]
    if not ((g["accept_len"][bad] == 0).all() and (g["out_tokens"][bad] == -1).all()
            and (g["path_nodes"][bad] == -1).all() and (g["accept_prob"][bad] == -1).all()):
        fails.append(("failed requests emit something", bad[:10].tolist()))
    rf = o["req_flag"]
    strict = ok & ((rf & oracle.FLAGS_STRICT) != 0)
    wide_only = ok & ((rf & oracle.FLAGS_WIDE) != 0) & ~strict
    deviations, flipped, worst = 0, 0, 0.0

    def alt(b, flip):
        return oracle.tree_sample_alt(ti.dtype, ti.target, ti.draft if sampled else None, ti.B, ti.N,
                                      ti.V, T, ti.node_tokens, ti.parents, ti.r if sampled else None,
                                      ti.u if sampled else None, int(b), flip, temperatures=temperatures)

    for b in np.nonzero(ok)[0]:
        L = int(g["accept_len"][b])
        ref = dict(accept_len=int(o["accept_len"][b]), path=o["path"][b], out_tokens=o["out_tokens"][b],
                   alpha=o["alpha"][b], mass=float(o["mass"][b]), req_flag=int(rf[b]))
        if L != ref["accept_len"] or not np.array_equal(g["path_nodes"][b], ref["path"]):
            if not rf[b] & (oracle.FLAG_ACCEPT_TIE | oracle.FLAG_ACCEPT_TIE_WIDE):
                fails.append(("path differs", int(b)))
                continue
            ref = alt(b, True)  # the other decision of the flagged test
            flipped += 1
            if L != ref["accept_len"] or not np.array_equal(g["path_nodes"][b], ref["path"]):
                fails.append(("path differs from both outcomes of the flagged test", int(b)))
                continue
        out = g["out_tokens"][b]
        if not np.array_equal(out[:L], ref["out_tokens"][:L]) or not (out[L + 1:] == -1).all():
            fails.append(("accepted tokens or padding differ", int(b)))
            continue
        t = int(out[L])
        if t != ref["out_tokens"][L]:
            full = ref if "draw_w" in ref else alt(b, False)
            flagged_draw = ref["req_flag"] & (oracle.FLAG_CDF_TIE | oracle.FLAG_CDF_TIE_WIDE)
            wmax = full["draw_wmax"] if ref["req_flag"] & oracle.FLAG_CDF_TIE_WIDE else None
            if not (sampled and flagged_draw and draw_admissible(
                    full["draw_w"], full["draw_cdf"], float(ti.u[b]), t, _tie_band(ref["mass"], True), wmax)):
                fails.append(("emitted token not admissible", int(b), t, int(ref["out_tokens"][L])))
                continue
            deviations += 1
        tested_g, tested_o = g["accept_prob"][b] >= 0, np.asarray(ref["alpha"]) >= 0
        if not np.array_equal(tested_g, tested_o):
            fails.append(("children tested differ", int(b)))
            continue
        da = np.abs(g["accept_prob"][b] - np.asarray(ref["alpha"]))[tested_o]
        if da.size:
            worst = max(worst, float(da.max()))
            if da.max() > PROB_TOL:
                fails.append(("alpha", int(b), float(da.max())))
        if abs(float(g["residual_mass"][b]) - ref["mass"]) > PROB_TOL:
            fails.append(("residual mass", int(b), float(g["residual_mass"][b]), ref["mass"]))
    return dict(requests=int(ok.size), errors=int((~ok).sum()), flagged=int((strict | wide_only).sum()),
                flagged_strict=int(strict.sum()), flagged_wide_only=int(wide_only.sum()),
                admissible_deviations=deviations, flipped_accept_ties=flipped,
                mean_accepted=float(g["accept_len"][ok].mean()) if ok.any() else 0.0,
                max_alpha_diff=worst, failures=fails)


def compare_walk(g: dict, o: dict, ti, temperature=None, temperatures=None) -> dict:
    """Asserts parity of a tree walk (see check_walk); returns the counts."""
    st = check_walk(g, o, ti, temperature, temperatures)
    assert not st["failures"], st["failures"][:10]
    return st
