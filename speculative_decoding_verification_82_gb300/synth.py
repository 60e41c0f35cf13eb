"""Seeded synthetic inputs for the target-side verification step of speculative decoding.

This module draws the *inputs* of the verification step and nothing else: target logits,
draft logits, draft tokens, the uniform variates the method consumes (r per draft position,
u per request), and draft-tree parent/token arrays.  It holds none of the verification
arithmetic (no temperature softmax, no acceptance ratio, no residual, no inverse CDF), so the
CUDA path and the CPU oracle can both be fed from it without sharing any of the method.

Every array comes from numpy's counter-based Philox generator, keyed by (seed, stream id), one
stream per array, filled in C order.  Consequently a configuration generated with a smaller
batch B is a prefix (the first B requests) of the same configuration at a larger B.

Uniform conventions (the pages only say "Uniform(0, 1)"):
  * r (acceptance test) lies in (0, 1]: r = (k + 1) * 2**-24, k uniform on [0, 2**24).
  * u (inverse-CDF resampling / bonus sampling) lies in [0, 1): u = k * 2**-24.
Both are exact in fp32, so the GPU and the oracle see identical values.

Draft tokens that the method expects to be drawn from the draft distribution q are sampled by
the Gumbel-max trick, x = argmax_i (d_i / T + G_i) with G_i standard Gumbel; this is the draft
mechanism's own sampling, done without evaluating a softmax.

Value distributions follow the five workloads of the verification benchmark (chain tiny,
chain small vocabulary, chain batched, greedy EAGLE-2-like tree, n-gram prompt lookup).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

U24 = 1.0 / float(1 << 24)

# Stream ids: one independent Philox key per drawn array.
_S_TARGET, _S_DRAFT, _S_SPIKE, _S_GUMBEL, _S_R, _S_U, _S_TREE, _S_PROMPT, _S_BOOST = range(1, 10)

DTYPES = ("f32", "bf16", "f16")


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=(int(seed) << 16) | int(stream)))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((b >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32, exact."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 values -> storage array of `dtype` ('f32' float32, 'bf16' uint16 bits, 'f16' float16)."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return to_bf16_bits(x)
    if dtype == "f16":
        return np.ascontiguousarray(x, dtype=np.float16)
    raise ValueError(dtype)


def decode(a: np.ndarray, dtype: str) -> np.ndarray:
    """Storage array -> fp32 values (exact)."""
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f32(a)
    if dtype == "f16":
        return np.asarray(a, dtype=np.float16).astype(np.float32)
    raise ValueError(dtype)


def uniform_r(seed: int, shape) -> np.ndarray:
    """Acceptance-test uniforms in (0, 1], exact multiples of 2**-24."""
    k = _rng(seed, _S_R).integers(0, 1 << 24, size=shape, dtype=np.int64)
    return ((k + 1) * U24).astype(np.float32)


def uniform_u(seed: int, shape) -> np.ndarray:
    """Resampling uniforms in [0, 1), exact multiples of 2**-24."""
    k = _rng(seed, _S_U).integers(0, 1 << 24, size=shape, dtype=np.int64)
    return (k * U24).astype(np.float32)


def gumbel_max_tokens(values: np.ndarray, temperature: float, rng: np.random.Generator) -> np.ndarray:
    """One token per row of `values` (..., V), drawn as argmax(values/T + Gumbel noise)."""
    flat = values.reshape(-1, values.shape[-1])
    out = np.empty(flat.shape[0], dtype=np.int32)
    t = float(temperature)
    for i in range(flat.shape[0]):
        g = rng.random(flat.shape[1])
        g = -np.log(-np.log(np.maximum(g, 1e-300)))
        out[i] = int(np.argmax(flat[i].astype(np.float64) / t + g))
    return out.reshape(values.shape[:-1])


@dataclass
class ChainInputs:
    """Inputs of one chain (or n-gram) verification call.

    target: [B][K+1][V] storage array (see `encode`); row k scores draft position k, row K is
            the bonus row.
    draft:  [B][K][V] storage array, or None for a one-hot (n-gram) or greedy draft.
    """

    name: str
    dtype: str
    B: int
    K: int
    V: int
    temperature: np.float32
    target: np.ndarray
    draft: np.ndarray | None
    draft_tokens: np.ndarray  # int32 [B][K]
    r: np.ndarray  # float32 [B][K], (0, 1]
    u: np.ndarray  # float32 [B], [0, 1)
    meta: dict = field(default_factory=dict)

    @property
    def logits_bytes(self) -> int:
        n = self.target.nbytes
        if self.draft is not None and float(self.temperature) > 0:
            n += self.draft.nbytes
        return n


@dataclass
class TreeInputs:
    """Inputs of one tree verification call.

    target:      [B][N+1][V] storage array; row n scores the children of node n.
    node_tokens: int32 [B][N+1]; node 0 is the root (its token is ignored).
    parents:     int32 [B][N+1]; parents[0] = -1, 0 <= parents[i] < i.
    Stochastic walks (temperature > 0) also carry
    draft:       [B][N+1][V] storage array; row n is the draft distribution the children of
                 node n were drawn from (rows of leaves are never read);
    r:           float32 [B][N+1], (0, 1]; r[b][c] is the uniform of child c's acceptance test;
    u:           float32 [B], [0, 1).
    """

    name: str
    dtype: str
    B: int
    N: int
    V: int
    target: np.ndarray
    node_tokens: np.ndarray
    parents: np.ndarray
    meta: dict = field(default_factory=dict)
    draft: np.ndarray | None = None
    r: np.ndarray | None = None
    u: np.ndarray | None = None
    temperature: np.float32 = np.float32(0.0)

    @property
    def logits_bytes(self) -> int:
        return self.target.nbytes

    @property
    def internal_nodes(self) -> np.ndarray:
        """bool [B][N+1]: nodes with at least one child (the rows whose draft side is read)."""
        out = np.zeros(self.parents.shape, dtype=bool)
        for b in range(self.B):
            par = self.parents[b, 1:]
            out[b, par[par >= 0]] = True
        return out


# ----------------------------------------------------------------------------------------------
# Workload 1: chain verify, tiny (distribution check).  One fixed set of logits per position,
# replicated over `trials` requests; draft tokens, r and u are fresh per trial.
# ----------------------------------------------------------------------------------------------
def chain_tiny(seed: int = 0, trials: int = 100_000, K: int = 5, V: int = 32,
               target_sigma: float = 2.0, draft_sigma: float = 1.0,
               temperature: float = 1.0) -> ChainInputs:
    T = np.float32(temperature)
    base_t = (_rng(seed, _S_TARGET).standard_normal((K + 1, V), dtype=np.float32)
              * np.float32(target_sigma))
    base_d = base_t[:K] + (_rng(seed, _S_DRAFT).standard_normal((K, V), dtype=np.float32)
                           * np.float32(draft_sigma))
    target = np.broadcast_to(base_t, (trials, K + 1, V)).copy()
    draft = np.broadcast_to(base_d, (trials, K, V)).copy()
    # fresh x_k ~ q_k per trial, vectorised Gumbel-max over the fixed draft rows
    g = _rng(seed, _S_GUMBEL).random((trials, K, V))
    g = -np.log(-np.log(np.maximum(g, 1e-300)))
    x = np.argmax(base_d[None].astype(np.float64) / float(T) + g, axis=-1).astype(np.int32)
    return ChainInputs("chain_tiny", "f32", trials, K, V, T, target, draft, x,
                       uniform_r(seed, (trials, K)), uniform_u(seed, (trials,)),
                       meta={"target_rows": base_t, "draft_rows": base_d})


# ----------------------------------------------------------------------------------------------
# Workload 2: chain verify, small vocabulary, bf16, T=0.7 (and greedy T=0).
# ----------------------------------------------------------------------------------------------
def chain_small_vocab(seed: int = 0, B: int = 1, K: int = 5, V: int = 32000,
                      temperature: float = 0.7, dtype: str = "bf16") -> ChainInputs:
    T = np.float32(temperature)
    t32 = _rng(seed, _S_TARGET).standard_normal((B, K + 1, V), dtype=np.float32) * np.float32(3.0)
    spike = _rng(seed, _S_SPIKE).integers(0, V, size=(B, K + 1))
    np.add.at(t32, (np.arange(B)[:, None], np.arange(K + 1)[None, :], spike), np.float32(8.0))
    d32 = t32[:, :K] + _rng(seed, _S_DRAFT).standard_normal((B, K, V), dtype=np.float32) * np.float32(1.5)
    target, draft = encode(t32, dtype), encode(d32, dtype)
    dvals = decode(draft, dtype)
    if float(T) > 0:
        x = gumbel_max_tokens(dvals, float(T), _rng(seed, _S_GUMBEL))
    else:
        x = np.argmax(dvals, axis=-1).astype(np.int32)  # greedy draft
    return ChainInputs("chain_small_vocab", dtype, B, K, V, T, target, draft, x.astype(np.int32),
                       uniform_r(seed, (B, K)), uniform_u(seed, (B,)))


# ----------------------------------------------------------------------------------------------
# Workload 3: chain verify, batched, fp32, V=128256, Zipf-spiked logits.
# ----------------------------------------------------------------------------------------------
def zipf_boosts(n: int = 20, hi: float = 10.0, lo: float = 2.0) -> np.ndarray:
    """Boost of the rank-r spike (r = 1..n): lo + (hi-lo) * (1/r - 1/n) / (1 - 1/n)."""
    rk = np.arange(1, n + 1, dtype=np.float64)
    return (lo + (hi - lo) * (1.0 / rk - 1.0 / n) / (1.0 - 1.0 / n)).astype(np.float32)


def chain_batched(seed: int = 0, B: int = 64, K: int = 5, V: int = 128256,
                  temperature: float = 1.0, dtype: str = "f32",
                  draft_tokens: str = "sample") -> ChainInputs:
    """`draft_tokens`: 'sample' draws x_k ~ q_k (Gumbel-max); 'argmax' takes the draft argmax
    (cheaper to generate at full size, used where only throughput matters)."""
    T = np.float32(temperature)
    t32 = _rng(seed, _S_TARGET).standard_normal((B, K + 1, V), dtype=np.float32) * np.float32(3.0)
    boosts = zipf_boosts()
    srng = _rng(seed, _S_SPIKE)
    for b in range(B):
        for k in range(K + 1):
            ids = srng.choice(V, size=boosts.size, replace=False)
            t32[b, k, ids] += boosts
    d32 = t32[:, :K] + _rng(seed, _S_DRAFT).standard_normal((B, K, V), dtype=np.float32) * np.float32(2.0)
    target, draft = encode(t32, dtype), encode(d32, dtype)
    del t32, d32
    if draft_tokens == "sample":
        x = gumbel_max_tokens(decode(draft, dtype), float(T), _rng(seed, _S_GUMBEL))
    else:
        x = np.argmax(decode(draft, dtype), axis=-1).astype(np.int32)
    return ChainInputs("chain_batched", dtype, B, K, V, T, target, draft, x.astype(np.int32),
                       uniform_r(seed, (B, K)), uniform_u(seed, (B,)))


# ----------------------------------------------------------------------------------------------
# Workload 4: greedy tree verify (EAGLE-2-like draft tree), bf16, V=128256.
# ----------------------------------------------------------------------------------------------
# 60 draft nodes in 6 levels; level sizes [10, 16, 12, 10, 6, 6]; per level, the lowest-index
# (highest-ranked) nodes of the previous level are expanded with the given branching factor.
TREE_LEVELS = ((1, 10), (4, 4), (4, 3), (5, 2), (3, 2), (3, 2))  # (expanded parents, children each)


def eagle_tree_parents(levels=TREE_LEVELS) -> np.ndarray:
    """Parent-index array of the draft tree, BFS numbering, node 0 = root, parents[0] = -1."""
    parents = [-1]
    prev = [0]
    for n_expand, branch in levels:
        cur = []
        for p in prev[:n_expand]:
            for _ in range(branch):
                parents.append(p)
                cur.append(len(parents) - 1)
        prev = cur
    return np.asarray(parents, dtype=np.int32)


def tree_greedy(seed: int = 0, B: int = 16, V: int = 128256, boost: float = 6.0,
                boost_frac: float = 0.7, dtype: str = "bf16",
                parents: np.ndarray | None = None, path_boost: float = 0.0) -> TreeInputs:
    """`path_boost` > 0 additionally boosts, per request, every node on the path from the root to
    one seeded deepest leaf (in its parent's row), so long paths occur."""
    par = eagle_tree_parents() if parents is None else np.asarray(parents, dtype=np.int32)
    N1 = par.size
    trng = _rng(seed, _S_TREE)
    tokens = np.zeros((B, N1), dtype=np.int32)
    for b in range(B):
        for p in range(N1):
            kids = np.nonzero(par == p)[0]
            if kids.size:
                tokens[b, kids] = trng.choice(V, size=kids.size, replace=False)  # distinct siblings
    t32 = _rng(seed, _S_TARGET).standard_normal((B, N1, V), dtype=np.float32) * np.float32(3.0)
    brng = _rng(seed, _S_BOOST)
    for b in range(B):
        for n in range(1, N1):
            if brng.random() < boost_frac:
                t32[b, par[n], tokens[b, n]] += np.float32(boost)
    if path_boost > 0:
        depth = np.zeros(N1, np.int64)
        for i in range(1, N1):
            depth[i] = depth[par[i]] + 1
        deepest = np.nonzero(depth == depth.max())[0]
        lrng = _rng(seed, _S_SPIKE)
        for b in range(B):
            v = int(lrng.choice(deepest))
            while v != 0:
                t32[b, par[v], tokens[b, v]] += np.float32(path_boost)
                v = int(par[v])
    return TreeInputs("tree_greedy", dtype, B, N1 - 1, V, encode(t32, dtype), tokens,
                      np.broadcast_to(par, (B, N1)).copy())


# ----------------------------------------------------------------------------------------------
# Workload 5: n-gram prompt-lookup verify (one-hot draft), bf16, V=151936, T=0.8.
# ----------------------------------------------------------------------------------------------
def ngram(seed: int = 0, B: int = 256, K: int = 5, V: int = 151936, temperature: float = 0.8,
          prompt_len: int = 2048, ngram_n: int = 4, boost: float = 5.0, boost_frac: float = 0.6,
          dtype: str = "bf16") -> ChainInputs:
    T = np.float32(temperature)
    prng = _rng(seed, _S_PROMPT)
    prompt = prng.integers(0, V, size=prompt_len).astype(np.int32)
    starts = prng.integers(0, prompt_len - ngram_n - K + 1, size=B)
    x = np.stack([prompt[s + ngram_n: s + ngram_n + K] for s in starts]).astype(np.int32)
    t32 = _rng(seed, _S_TARGET).standard_normal((B, K + 1, V), dtype=np.float32) * np.float32(3.0)
    hit = _rng(seed, _S_BOOST).random((B, K)) < boost_frac
    bb, kk = np.nonzero(hit)
    t32[bb, kk, x[bb, kk]] += np.float32(boost)
    return ChainInputs("ngram", dtype, B, K, V, T, encode(t32, dtype), None, x,
                       uniform_r(seed, (B, K)), uniform_u(seed, (B,)),
                       meta={"prompt": prompt, "starts": starts})


# ----------------------------------------------------------------------------------------------
# Stochastic tree verify (T > 0 over an EAGLE-2-like tree): the tree of workload 4 with the
# value recipe of workload 3 (target ~ N(0, 3^2) with Zipf-shaped spikes, draft = target +
# N(0, 2^2)); the children of node n are independent draws from the draft distribution of row n.
# ----------------------------------------------------------------------------------------------
def _draw_children(par: np.ndarray, drow, T: float, rng: np.random.Generator) -> np.ndarray:
    """Tokens of one request's nodes: the children of node n drawn independently from the draft
    distribution of row n (Gumbel-max over drow(n), a float32 [V] row)."""
    tokens = np.zeros(par.size, dtype=np.int32)
    for p in range(par.size):
        kids = np.nonzero(par == p)[0]
        if kids.size:
            d = drow(p).astype(np.float64) / T
            g = rng.random((kids.size, d.size))
            g = -np.log(-np.log(np.maximum(g, 1e-300)))
            tokens[kids] = np.argmax(d[None, :] + g, axis=1)
    return tokens


def tree_sample(seed: int = 0, B: int = 16, V: int = 128256, temperature: float = 1.0,
                dtype: str = "bf16", parents: np.ndarray | None = None,
                draft_sigma: float = 2.0) -> TreeInputs:
    T = np.float32(temperature)
    par = eagle_tree_parents() if parents is None else np.asarray(parents, dtype=np.int32)
    N1 = par.size
    t32 = _rng(seed, _S_TARGET).standard_normal((B, N1, V), dtype=np.float32) * np.float32(3.0)
    boosts = zipf_boosts()
    srng = _rng(seed, _S_SPIKE)
    ns = min(boosts.size, V)  # a vocabulary smaller than the spike count takes the largest ones
    for b in range(B):
        for n in range(N1):
            t32[b, n, srng.choice(V, size=ns, replace=False)] += boosts[:ns]
    d32 = t32 + _rng(seed, _S_DRAFT).standard_normal((B, N1, V), dtype=np.float32) * np.float32(draft_sigma)
    target, draft = encode(t32, dtype), encode(d32, dtype)
    del t32, d32
    grng = _rng(seed, _S_GUMBEL)
    tokens = np.stack([_draw_children(par, lambda n, b=b: decode(draft[b, n], dtype), float(T), grng)
                       for b in range(B)])
    return TreeInputs("tree_sample", dtype, B, N1 - 1, V, target, tokens,
                      np.broadcast_to(par, (B, N1)).copy(), draft=draft,
                      r=uniform_r(seed, (B, N1)), u=uniform_u(seed, (B,)), temperature=T)


def tree_sample_tiny(seed: int = 0, trials: int = 100_000, V: int = 8, branching=(3, 2),
                     temperature: float = 1.0, target_sigma: float = 2.0,
                     draft_sigma: float = 1.0) -> TreeInputs:
    """Distribution check of the stochastic walk: a two-level tree whose rows depend only on the
    token prefix (root; token a at depth 1; tokens (a, b) at depth 2), so that the emitted token
    after a prefix must follow that prefix's target row.  Fresh children tokens (independent
    draws from the parent's draft row), r and u per trial; one fixed set of rows."""
    T = float(temperature)
    m1, m2 = branching
    rt = _rng(seed, _S_TARGET)
    rd = _rng(seed, _S_DRAFT)
    t0 = rt.standard_normal(V, dtype=np.float32) * np.float32(target_sigma)
    t1 = rt.standard_normal((V, V), dtype=np.float32) * np.float32(target_sigma)
    t2 = rt.standard_normal((V, V, V), dtype=np.float32) * np.float32(target_sigma)
    d0 = t0 + rd.standard_normal(V, dtype=np.float32) * np.float32(draft_sigma)
    d1 = t1 + rd.standard_normal((V, V), dtype=np.float32) * np.float32(draft_sigma)
    d2 = t2 + rd.standard_normal((V, V, V), dtype=np.float32) * np.float32(draft_sigma)
    par = [-1] + [0] * m1
    for i in range(m1):
        par += [1 + i] * m2
    par = np.asarray(par, dtype=np.int32)
    N1 = par.size
    g = _rng(seed, _S_GUMBEL)

    def gumbel(shape):
        x = g.random(shape)
        return -np.log(-np.log(np.maximum(x, 1e-300)))

    a = np.argmax(d0.astype(np.float64)[None, None, :] / T + gumbel((trials, m1, V)), axis=-1)
    bt = np.argmax(d1[a].astype(np.float64)[:, :, None, :] / T + gumbel((trials, m1, m2, V)), axis=-1)
    tokens = np.zeros((trials, N1), dtype=np.int32)
    tokens[:, 1: 1 + m1] = a
    tokens[:, 1 + m1:] = bt.reshape(trials, m1 * m2)
    target = np.empty((trials, N1, V), dtype=np.float32)
    draft = np.empty((trials, N1, V), dtype=np.float32)
    target[:, 0], draft[:, 0] = t0, d0
    target[:, 1: 1 + m1], draft[:, 1: 1 + m1] = t1[a], d1[a]
    aa = np.repeat(a, m2, axis=1)
    bb = bt.reshape(trials, m1 * m2)
    target[:, 1 + m1:], draft[:, 1 + m1:] = t2[aa, bb], d2[aa, bb]
    return TreeInputs("tree_sample_tiny", "f32", trials, N1 - 1, V, target, tokens,
                      np.broadcast_to(par, (trials, N1)).copy(),
                      meta={"t0": t0, "t1": t1, "t2": t2, "d0": d0, "d1": d1},
                      draft=draft, r=uniform_r(seed, (trials, N1)), u=uniform_u(seed, (trials,)),
                      temperature=np.float32(T))


def ngram_contexts(seed: int = 0, B: int = 256, K: int = 5, V: int = 151936, prompt_len: int = 2048,
                   ngram_n: int = 4) -> tuple[np.ndarray, np.ndarray]:
    """The contexts behind the n-gram workload: per request, the prompt followed by the 4 prompt
    tokens at the request's seeded start s (the generated text repeating a prompt 4-gram), so
    that prompt lookup proposes prompt[s + 4 .. s + 4 + K), the workload's drafts.  Same streams
    as `ngram`.  Returns ctx [B][prompt_len + ngram_n] int32 and the lengths [B]."""
    prng = _rng(seed, _S_PROMPT)
    prompt = prng.integers(0, V, size=prompt_len).astype(np.int32)
    starts = prng.integers(0, prompt_len - ngram_n - K + 1, size=B)
    ctx = np.empty((B, prompt_len + ngram_n), dtype=np.int32)
    ctx[:, :prompt_len] = prompt
    for b, s0 in enumerate(starts):
        ctx[b, prompt_len:] = prompt[s0: s0 + ngram_n]
    return ctx, np.full(B, prompt_len + ngram_n, dtype=np.int32)


def kv_compact_case(seed: int = 0, B: int = 16, caches: int = 160, row_bytes: int = 2048,
                    parents: np.ndarray | None = None, deepest: bool = True) -> dict:
    """Inputs of accepted-path KV compaction: the draft tree of workload 4 (or `parents`), one
    accepted path per request (from the root to a seeded deepest node, or to any seeded node), the
    slots of request b's nodes b * (N + 1) + n, and `caches` caches of random bytes with one row
    per slot.  The default sizes are those of Llama-3.3-70B (the page's serving example: 80 layers,
    8 KV heads of 128 bf16 values: 160 K/V caches of 2048-byte rows)."""
    par = eagle_tree_parents() if parents is None else np.asarray(parents, dtype=np.int32)
    N1 = par.size
    depth = np.zeros(N1, np.int64)
    for i in range(1, N1):
        depth[i] = depth[par[i]] + 1
    rng = _rng(seed, _S_TREE)
    pool = np.nonzero(depth == depth.max())[0] if deepest else np.arange(N1)
    path = np.full((B, N1), -1, np.int32)
    accept_len = np.zeros(B, np.int32)
    for b in range(B):
        v = int(rng.choice(pool))
        chain = [v]
        while chain[-1] != 0:
            chain.append(int(par[chain[-1]]))
        chain = chain[::-1]
        path[b, : len(chain)] = chain
        accept_len[b] = len(chain) - 1
    slots = (np.arange(B, dtype=np.int32)[:, None] * N1 + np.arange(N1, dtype=np.int32)[None, :]).astype(np.int32)
    data = _rng(seed, _S_TARGET).integers(0, 256, size=(caches, B * N1, row_bytes), dtype=np.uint8)
    return dict(caches=data, slots=slots, parents=np.broadcast_to(par, (B, N1)).copy(),
                accept_len=accept_len, path=path)
