"""CPU oracle for the target-side verification step of speculative decoding.

TEST INFRASTRUCTURE: a plain scalar C reference (``spec_oracle.c``, double precision) plus this
ctypes shim.  Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU baseline leg
may import it.  It does not import the CUDA package and shares no code with it; both are fed
from the seeded input generators.

Parity pinning: every function here is pinned by ``tests/test_oracle_*.py`` against hand-worked
cases, closed forms, the invariance theorem (chi-squared), brute force and library routines.
The conventions that the pages leave open (uniform ranges, tie-breaks, the bonus draw, the tree
layout) are readings, listed in the oracle source header; parity on those is "GPU equals oracle",
not "equals the pages".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from ctypes import POINTER, c_double, c_float, c_int, c_size_t, c_void_p

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "spec_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "libspec_oracle.so")

DTYPE_CODE = {"f32": 0, "bf16": 1, "f16": 2}
FLAG_ACCEPT_TIE, FLAG_CDF_TIE, FLAG_ZERO_RESIDUAL = 1, 2, 4
# the widened tie tier (reading R10 / R14): within tol / S (tol / R) of a boundary but not within tol
FLAG_CDF_TIE_WIDE, FLAG_ACCEPT_TIE_WIDE = 8, 16
FLAGS_STRICT = FLAG_ACCEPT_TIE | FLAG_CDF_TIE
FLAGS_WIDE = FLAG_ACCEPT_TIE_WIDE | FLAG_CDF_TIE_WIDE
ERR_BAD_TOKEN, ERR_NONFINITE, ERR_BAD_TREE, ERR_BAD_TEMP = 1, 2, 8, 16
DEFAULT_TOL = 1e-6

_lock = threading.Lock()
_lib = None


def build(src: str = SRC, out: str = LIB, extra_flags=()) -> str:
    """Compile the oracle with gcc (plain C, no fused multiply-add, no fast math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           *extra_flags, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _needs_build(lib: str, src: str) -> bool:
    return not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src)


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    I, D, F, P = c_int, c_double, c_float, c_void_p
    lib.oracle_softmax.argtypes = [P, I, D, P]
    lib.oracle_softmax.restype = I
    lib.oracle_argmax.argtypes = [P, I]
    lib.oracle_argmax.restype = I
    lib.oracle_inverse_cdf.argtypes = [P, I, D, D, POINTER(c_double), POINTER(c_int)]
    lib.oracle_inverse_cdf.restype = I
    lib.oracle_verify_probs.argtypes = [I, I, P, P, P, P, F, D, P, P, P, P, P, P, P]
    lib.oracle_verify_probs.restype = None
    lib.oracle_verify_ngram_direct.argtypes = [I, I, P, P, P, F, D, P, P, P, P, P, P, P]
    lib.oracle_verify_ngram_direct.restype = None
    lib.oracle_verify_chain.argtypes = [I, P, P, I, I, I, F, P, P, P, P, D, I, I,
                                        P, P, P, P, P, P, P, P]
    lib.oracle_verify_chain.restype = None
    lib.oracle_verify_ngram.argtypes = [I, P, I, I, I, F, P, P, P, P, D, I, I,
                                        P, P, P, P, P, P, P, P]
    lib.oracle_verify_ngram.restype = None
    lib.oracle_tree_check.argtypes = [I, I, P, P]
    lib.oracle_tree_check.restype = I
    lib.oracle_tree_walk.argtypes = [I, P, P, P, P, P, P]
    lib.oracle_tree_walk.restype = None
    lib.oracle_tree_bruteforce.argtypes = [I, P, P, P, POINTER(c_int)]
    lib.oracle_tree_bruteforce.restype = I
    lib.oracle_verify_tree_greedy.argtypes = [I, P, I, I, I, P, P, I, I, P, P, P, P, P]
    lib.oracle_verify_tree_greedy.restype = None
    lib.oracle_tree_sample_probs.argtypes = [I, I, P, P, P, P, P, F, D, I, P, P, P, P, P, P, P, P, P]
    lib.oracle_tree_sample_probs.restype = None
    lib.oracle_verify_tree_sample.argtypes = [I, P, P, I, I, I, F, P, P, P, P, P, D, I, I,
                                              P, P, P, P, P, P, P]
    lib.oracle_verify_tree_sample.restype = None
    lib.oracle_chain_draw_rows.argtypes = [I, P, P, I, I, I, F, P, I, D, P, P, P]
    lib.oracle_chain_draw_rows.restype = I
    lib.oracle_tree_sample_alt.argtypes = [I, P, P, I, I, F, P, P, P, P, P, D, I, I,
                                           P, P, P, P, P, P, P, P, P]
    lib.oracle_tree_sample_alt.restype = I
    lib.oracle_ngram_draft.argtypes = [P, I, I, I, I, P, P, P, P]
    lib.oracle_ngram_draft.restype = None
    lib.oracle_ngram_draft_batch.argtypes = [P, P, I, I, I, I, I, I, I, P, P, P, P, P]
    lib.oracle_ngram_draft_batch.restype = None
    lib.oracle_kv_compact.argtypes = [P, I, P, I, P]
    lib.oracle_kv_compact.restype = None
    lib.oracle_kv_compact_batch.argtypes = [P, I, ctypes.c_longlong, I, I, I, P, P, P, P, P]
    lib.oracle_kv_compact_batch.restype = None
    lib.oracle_load.argtypes = [P, I, c_size_t]
    lib.oracle_load.restype = D
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library.  `path` loads a specific build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build(LIB, SRC):
                build()
            _lib = _bind(ctypes.CDLL(LIB))
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------------------ primitives ----
def softmax(logits, T: float, lib=None) -> tuple[np.ndarray, int]:
    lib = lib or load()
    l = _c(logits, np.float64)
    p = np.empty_like(l)
    e = lib.oracle_softmax(_p(l), l.size, float(T), _p(p))
    return p, e


def argmax(logits, lib=None) -> int:
    lib = lib or load()
    l = _c(logits, np.float64)
    return lib.oracle_argmax(_p(l), l.size)


def inverse_cdf(w, u: float, tol: float = DEFAULT_TOL, lib=None) -> tuple[int, float, int]:
    lib = lib or load()
    w = _c(w, np.float64)
    S, fl = c_double(), c_int()
    i = lib.oracle_inverse_cdf(_p(w), w.size, float(u), tol, ctypes.byref(S), ctypes.byref(fl))
    return i, S.value, fl.value


def _alloc_chain_out(B: int, K: int) -> dict:
    return dict(num_accepted=np.zeros(B, np.int32), out_tokens=np.zeros((B, K + 1), np.int32),
                alpha=np.zeros((B, K), np.float64), cand=np.zeros((B, K + 1), np.int32),
                mass=np.zeros((B, K + 1), np.float64), pos_flag=np.zeros((B, K + 1), np.int32),
                req_flag=np.zeros(B, np.int32), err=np.zeros(B, np.int32))


def verify_probs(p, q, x, r, u, tol: float = DEFAULT_TOL, lib=None) -> dict:
    """One request from probability rows p [K+1][V], q [K][V]."""
    lib = lib or load()
    p = _c(p, np.float64)
    K = p.shape[0] - 1
    V = p.shape[1]
    q = _c(q, np.float64).reshape(K, V) if K else np.zeros((0, V))
    x, r = _c(x, np.int32).reshape(K), _c(r, np.float32).reshape(K)
    o = _alloc_chain_out(1, K)
    lib.oracle_verify_probs(K, V, _p(p), _p(q), _p(x), _p(r), float(u), tol,
                            _p(o["num_accepted"]), _p(o["out_tokens"]), _p(o["alpha"]),
                            _p(o["cand"]), _p(o["mass"]), _p(o["pos_flag"]), _p(o["req_flag"]))
    return {k: v[0] for k, v in o.items() if k != "err"}


def verify_ngram_direct(p, x, r, u, tol: float = DEFAULT_TOL, lib=None) -> dict:
    lib = lib or load()
    p = _c(p, np.float64)
    K, V = p.shape[0] - 1, p.shape[1]
    x, r = _c(x, np.int32).reshape(K), _c(r, np.float32).reshape(K)
    o = _alloc_chain_out(1, K)
    lib.oracle_verify_ngram_direct(K, V, _p(p), _p(x), _p(r), float(u), tol,
                                   _p(o["num_accepted"]), _p(o["out_tokens"]), _p(o["alpha"]),
                                   _p(o["cand"]), _p(o["mass"]), _p(o["pos_flag"]),
                                   _p(o["req_flag"]))
    return {k: v[0] for k, v in o.items() if k != "err"}


# --------------------------------------------------------------------------- whole calls ----
def _ranges(B: int, threads: int):
    threads = max(1, min(threads, B))
    step = (B + threads - 1) // threads
    return [(b, min(B, b + step)) for b in range(0, B, step)]


def _run_threaded(fn, B: int, threads: int):
    """ctypes releases the GIL during the call, so request ranges run on separate cores."""
    rngs = _ranges(B, threads)
    if len(rngs) <= 1:
        for b0, b1 in rngs:
            fn(b0, b1)
        return
    ts = [threading.Thread(target=fn, args=rg) for rg in rngs]
    for t in ts:
        t.start()
    for t in ts:
        t.join()


def verify_chain(dtype: str, target, draft, B: int, K: int, V: int, T: float, draft_tokens, r, u,
                 tol: float = DEFAULT_TOL, threads: int = 1, requests=None, lib=None,
                 temperatures=None) -> dict:
    """Chain verification of `B` requests (or only the index range `requests`=(b0, b1));
    `temperatures` [B] sets each request's own temperature (R18)."""
    lib = lib or load()
    target = np.ascontiguousarray(target)
    draft_a = np.ascontiguousarray(draft) if draft is not None else None
    draft_p = _p(draft_a) if draft_a is not None else None
    x = _c(draft_tokens, np.int32)
    rr = _c(r, np.float32) if r is not None else np.zeros((B, K), np.float32)
    uu = _c(u, np.float32) if u is not None else np.zeros(B, np.float32)
    tt = _c(temperatures, np.float32) if temperatures is not None else None
    o = _alloc_chain_out(B, K)
    keep = (target, draft_a, tt)

    def run(b0, b1):
        lib.oracle_verify_chain(DTYPE_CODE[dtype], _p(target), draft_p, B, K, V, float(T),
                                _p(tt) if tt is not None else None, _p(x),
                                _p(rr), _p(uu), tol, b0, b1, *(_p(o[k]) for k in (
                                    "num_accepted", "out_tokens", "alpha", "cand", "mass",
                                    "pos_flag", "req_flag", "err")))

    if requests is not None:
        run(*requests)
    else:
        _run_threaded(run, B, threads)
    del keep
    return o


def verify_ngram(dtype: str, target, B: int, K: int, V: int, T: float, draft_tokens, r, u,
                 tol: float = DEFAULT_TOL, threads: int = 1, requests=None, lib=None,
                 temperatures=None) -> dict:
    """n-gram (one-hot draft) verification; `temperatures` as in `verify_chain`."""
    lib = lib or load()
    target = np.ascontiguousarray(target)
    x = _c(draft_tokens, np.int32)
    rr = _c(r, np.float32) if r is not None else np.zeros((B, K), np.float32)
    uu = _c(u, np.float32) if u is not None else np.zeros(B, np.float32)
    tt = _c(temperatures, np.float32) if temperatures is not None else None
    o = _alloc_chain_out(B, K)

    def run(b0, b1):
        lib.oracle_verify_ngram(DTYPE_CODE[dtype], _p(target), B, K, V, float(T),
                                _p(tt) if tt is not None else None, _p(x), _p(rr),
                                _p(uu), tol, b0, b1, *(_p(o[k]) for k in (
                                    "num_accepted", "out_tokens", "alpha", "cand", "mass",
                                    "pos_flag", "req_flag", "err")))

    if requests is not None:
        run(*requests)
    else:
        _run_threaded(run, B, threads)
    return o


def chain_draw_rows(dtype: str, target, draft, B: int, K: int, V: int, T: float, draft_tokens,
                    b: int, ngram: bool = False, tol: float = DEFAULT_TOL, lib=None) -> dict:
    """The draws of request b of a chain (or n-gram) call, for checking a flagged tie:
    w [K+1][V], the weights each position's draw uses (residual, bonus row, or p after an empty
    residual); cdf [K+1][V], their normalised cumulative sums (token t is drawn at k for u in
    [cdf[k][t-1], cdf[k][t])); wmax [K+1][V], each token's largest weight within the widened
    tier's precision (R10); err, the request's error bits."""
    lib = lib or load()
    target = np.ascontiguousarray(target)
    dr = np.ascontiguousarray(draft) if (draft is not None and not ngram) else None
    x = _c(draft_tokens, np.int32)
    w = np.zeros((K + 1, V), np.float64)
    cdf = np.zeros((K + 1, V), np.float64)
    wmax = np.zeros((K + 1, V), np.float64)
    e = lib.oracle_chain_draw_rows(DTYPE_CODE[dtype], _p(target), _p(dr) if dr is not None else None,
                                   1 if ngram else 0, K, V, float(T), _p(x), int(b), tol, _p(w), _p(cdf),
                                   _p(wmax))
    return dict(w=w, cdf=cdf, wmax=wmax, err=int(e))


def tree_sample_alt(dtype: str, target, draft, B: int, N: int, V: int, T: float, node_tokens,
                    parents, r, u, b: int, flip: bool, tol: float = DEFAULT_TOL, temperatures=None,
                    lib=None) -> dict:
    """Request b of `verify_tree_sample`, with the first flagged accept test decided the other way
    when `flip`, plus the final draw's weights `draw_w` and normalised CDF `draw_cdf` ([V])."""
    lib = lib or load()
    target = np.ascontiguousarray(target)
    dr = np.ascontiguousarray(draft) if draft is not None else None
    tk, pa = _c(node_tokens, np.int32), _c(parents, np.int32)
    N1 = N + 1
    rr = _c(r, np.float32) if r is not None else np.zeros((B, N1), np.float32)
    uu = _c(u, np.float32) if u is not None else np.zeros(B, np.float32)
    tt = _c(temperatures, np.float32) if temperatures is not None else None
    L, fl = np.zeros(1, np.int32), np.zeros(1, np.int32)
    path, out = np.zeros(N1, np.int32), np.zeros(N1, np.int32)
    alpha, mass = np.zeros(N1, np.float64), np.zeros(1, np.float64)
    dw, dc, dm = (np.zeros(max(V, 1), np.float64) for _ in range(3))
    e = lib.oracle_tree_sample_alt(DTYPE_CODE[dtype], _p(target), _p(dr) if dr is not None else None,
                                   N, V, float(T), _p(tt) if tt is not None else None, _p(tk), _p(pa),
                                   _p(rr), _p(uu), tol, int(b), 1 if flip else 0, _p(L), _p(path),
                                   _p(out), _p(alpha), _p(mass), _p(fl), _p(dw), _p(dc), _p(dm))
    return dict(accept_len=int(L[0]), path=path, out_tokens=out, alpha=alpha, mass=float(mass[0]),
                req_flag=int(fl[0]), err=int(e), draw_w=dw, draw_cdf=dc, draw_wmax=dm)


def tree_walk(parents, tokens, amax, lib=None) -> dict:
    lib = lib or load()
    pa, tk, am = _c(parents, np.int32), _c(tokens, np.int32), _c(amax, np.int32)
    N1 = pa.size
    L = np.zeros(1, np.int32)
    path, out = np.zeros(N1, np.int32), np.zeros(N1, np.int32)
    lib.oracle_tree_walk(N1, _p(pa), _p(tk), _p(am), _p(L), _p(path), _p(out))
    return dict(accept_len=int(L[0]), path=path, out_tokens=out)


def tree_bruteforce(parents, tokens, amax, lib=None) -> tuple[int, int]:
    lib = lib or load()
    pa, tk, am = _c(parents, np.int32), _c(tokens, np.int32), _c(amax, np.int32)
    d = c_int()
    v = lib.oracle_tree_bruteforce(pa.size, _p(pa), _p(tk), _p(am), ctypes.byref(d))
    return v, d.value


def tree_check(parents, tokens, V: int, lib=None) -> int:
    lib = lib or load()
    pa, tk = _c(parents, np.int32), _c(tokens, np.int32)
    return lib.oracle_tree_check(pa.size, V, _p(pa), _p(tk))


def verify_tree_greedy(dtype: str, target, B: int, N: int, V: int, node_tokens, parents,
                       threads: int = 1, requests=None, lib=None) -> dict:
    lib = lib or load()
    target = np.ascontiguousarray(target)
    tk, pa = _c(node_tokens, np.int32), _c(parents, np.int32)
    N1 = N + 1
    o = dict(accept_len=np.zeros(B, np.int32), path=np.zeros((B, N1), np.int32),
             out_tokens=np.zeros((B, N1), np.int32), amax=np.zeros((B, N1), np.int32),
             err=np.zeros(B, np.int32))

    def run(b0, b1):
        lib.oracle_verify_tree_greedy(DTYPE_CODE[dtype], _p(target), B, N, V, _p(tk), _p(pa), b0,
                                      b1, _p(o["accept_len"]), _p(o["path"]),
                                      _p(o["out_tokens"]), _p(o["amax"]), _p(o["err"]))

    if requests is not None:
        run(*requests)
    else:
        _run_threaded(run, B, threads)
    return o


def tree_sample_probs(p, q, parents, tokens, r, u, tol: float = DEFAULT_TOL, lib=None,
                      flip: bool = False) -> dict:
    """One request of the stochastic tree walk from probability rows p, q [N+1][V]; with `flip`
    the first flagged accept test is decided the other way.  Also returns the final draw's
    weights `draw_w` and normalised CDF `draw_cdf` (zeros when the walk ends without a draw)."""
    lib = lib or load()
    p, q = _c(p, np.float64), _c(q, np.float64)
    N1, V = p.shape
    pa, tk, rr = _c(parents, np.int32), _c(tokens, np.int32), _c(r, np.float32)
    L, fl = np.zeros(1, np.int32), np.zeros(1, np.int32)
    path, out = np.zeros(N1, np.int32), np.zeros(N1, np.int32)
    alpha, mass = np.zeros(N1, np.float64), np.zeros(1, np.float64)
    dw, dc, dm = (np.zeros(V, np.float64) for _ in range(3))
    lib.oracle_tree_sample_probs(N1, V, _p(p), _p(q), _p(pa), _p(tk), _p(rr), float(u), tol,
                                 1 if flip else 0, _p(L), _p(path), _p(out), _p(alpha), _p(mass),
                                 _p(fl), _p(dw), _p(dc), _p(dm))
    return dict(accept_len=int(L[0]), path=path, out_tokens=out, alpha=alpha,
                mass=float(mass[0]), req_flag=int(fl[0]), draw_w=dw, draw_cdf=dc, draw_wmax=dm)


def verify_tree_sample(dtype: str, target, draft, B: int, N: int, V: int, T: float, node_tokens,
                       parents, r, u, tol: float = DEFAULT_TOL, threads: int = 1, requests=None,
                       lib=None, temperatures=None) -> dict:
    """Tree verification by walking: stochastic (T > 0) or greedy (T == 0) on visited rows;
    `temperatures` [B] sets each request's own temperature (R18)."""
    lib = lib or load()
    target = np.ascontiguousarray(target)
    draft_p = _p(np.ascontiguousarray(draft)) if draft is not None else None
    tk, pa = _c(node_tokens, np.int32), _c(parents, np.int32)
    N1 = N + 1
    rr = _c(r, np.float32) if r is not None else np.zeros((B, N1), np.float32)
    uu = _c(u, np.float32) if u is not None else np.zeros(B, np.float32)
    tt = _c(temperatures, np.float32) if temperatures is not None else None
    o = dict(accept_len=np.zeros(B, np.int32), path=np.zeros((B, N1), np.int32),
             out_tokens=np.zeros((B, N1), np.int32), alpha=np.zeros((B, N1), np.float64),
             mass=np.zeros(B, np.float64), req_flag=np.zeros(B, np.int32),
             err=np.zeros(B, np.int32))
    keep = (target, draft, tt)

    def run(b0, b1):
        lib.oracle_verify_tree_sample(DTYPE_CODE[dtype], _p(target), draft_p, B, N, V, float(T),
                                      _p(tt) if tt is not None else None, _p(tk), _p(pa), _p(rr),
                                      _p(uu), tol, b0, b1,
                                      *(_p(o[k]) for k in ("accept_len", "path", "out_tokens",
                                                           "alpha", "mass", "req_flag", "err")))

    if requests is not None:
        run(*requests)
    else:
        _run_threaded(run, B, threads)
    del keep
    return o


def ngram_draft(ctx, K: int, n_max: int = 4, n_min: int = 1, lib=None) -> dict:
    """Prompt lookup draft of one context (R16)."""
    lib = lib or load()
    c = _c(ctx, np.int32).reshape(-1)
    d = np.zeros(max(K, 1), np.int32)
    ln, mn, me = c_int(), c_int(), c_int()
    lib.oracle_ngram_draft(_p(c), c.size, n_max, n_min, K, _p(d), ctypes.byref(ln), ctypes.byref(mn),
                           ctypes.byref(me))
    return dict(draft=d[:K], draft_len=ln.value, match_n=mn.value, match_end=me.value)


def ngram_draft_batch(ctx, ctx_len, K: int, n_max: int = 4, n_min: int = 1, threads: int = 1,
                      lib=None) -> dict:
    """Prompt lookup drafts of B contexts ctx [B][Lmax] with lengths ctx_len [B]."""
    lib = lib or load()
    c, cl = _c(ctx, np.int32), _c(ctx_len, np.int32)
    B, Lmax = c.shape
    o = dict(draft=np.zeros((B, K), np.int32), draft_len=np.zeros(B, np.int32),
             match_n=np.zeros(B, np.int32), match_end=np.zeros(B, np.int32), err=np.zeros(B, np.int32))

    def run(b0, b1):
        lib.oracle_ngram_draft_batch(_p(c), _p(cl), B, Lmax, n_max, n_min, K, b0, b1,
                                     *(_p(o[k]) for k in ("draft", "draft_len", "match_n",
                                                          "match_end", "err")))

    _run_threaded(run, B, threads)
    return o


def kv_compact(cache, slots, accept_len: int, path, lib=None) -> np.ndarray:
    """One request, one cache [num_slots][row_bytes] (uint8): returns the compacted copy (R17)."""
    lib = lib or load()
    out = np.array(cache, dtype=np.uint8, copy=True, order="C")
    sl, pt = _c(slots, np.int32), _c(path, np.int32)
    lib.oracle_kv_compact(_p(out), out.shape[1], _p(sl), int(accept_len), _p(pt))
    return out


def kv_compact_batch(caches, slots, parents, accept_len, path, lib=None) -> tuple[np.ndarray, np.ndarray]:
    """caches [C][num_slots][row_bytes] uint8 (copied), slots / parents / path [B][N1],
    accept_len [B]: the compacted caches and the per-request error bits."""
    lib = lib or load()
    out = np.array(caches, dtype=np.uint8, copy=True, order="C")
    C, S, W = out.shape
    sl, pa, pt, al = (_c(a, np.int32) for a in (slots, parents, path, accept_len))
    B, N1 = sl.shape
    err = np.zeros(B, np.int32)
    lib.oracle_kv_compact_batch(_p(out), C, S, W, B, N1, _p(sl), _p(pa), _p(al), _p(pt), _p(err))
    return out, err


def load_elems(storage: np.ndarray, dtype: str, lib=None) -> np.ndarray:
    """Widen a storage array to float64 through the oracle's own converter (for tests)."""
    lib = lib or load()
    a = np.ascontiguousarray(storage)
    return np.array([lib.oracle_load(_p(a), DTYPE_CODE[dtype], i) for i in range(a.size)])
