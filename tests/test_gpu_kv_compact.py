"""GPU parity of accepted-path KV-cache compaction (spec_kv_compact) against the CPU oracle:
random trees, paths and slot permutations, several caches and row sizes, invalid requests, the
benchmark configuration (160 caches of 2048-byte rows, deepest paths of the 61-node tree) and
the verification-then-compaction sequence on the greedy tree workload; also stream order around
each call, eagerly and in a replayed CUDA graph."""

import numpy as np
import pytest
import torch

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


def _run(caches, slots, parents, accept_len, path):
    dev = [torch.from_numpy(np.ascontiguousarray(c)).cuda() for c in caches]
    err = binding.spec_kv_compact(dev, parity.i32(slots), parity.i32(parents), parity.i32(accept_len),
                                  parity.i32(path))
    torch.cuda.synchronize()
    return np.stack([d.cpu().numpy() for d in dev]), err.cpu().numpy()


@pytest.mark.parametrize("row_bytes,C", [(16, 1), (48, 3), (2048, 4), (4096, 2), (4112, 1)])
def test_random_paths_and_slots(row_bytes, C):
    rng = np.random.default_rng(row_bytes + C)
    B, N1 = 40, int(rng.integers(2, 30))
    parents = np.zeros((B, N1), np.int32)
    path = np.full((B, N1), -1, np.int32)
    al = np.zeros(B, np.int32)
    for b in range(B):
        par, _ = pins.random_tree(rng, N1, 50)
        parents[b] = par
        v = int(rng.integers(0, N1))
        chain = [v]
        while chain[-1] != 0:
            chain.append(int(par[chain[-1]]))
        chain = chain[::-1]
        path[b, : len(chain)] = chain
        al[b] = len(chain) - 1
    S = B * N1 + 17
    slots = rng.permutation(S)[: B * N1].reshape(B, N1).astype(np.int32)  # disjoint, scattered
    caches = rng.integers(0, 256, (C, S, row_bytes), dtype=np.uint8)
    g, gerr = _run(caches, slots, parents, al, path)
    o, oerr = oracle.kv_compact_batch(caches, slots, parents, al, path)
    assert np.array_equal(gerr, oerr) and (oerr == 0).all()
    assert np.array_equal(g, o)


def test_invalid_requests_are_left_untouched():
    kc = synth.kv_compact_case(seed=3, B=6, caches=2, row_bytes=64)
    al, path, slots = kc["accept_len"].copy(), kc["path"].copy(), kc["slots"].copy()
    al[1] = kc["parents"].shape[1]       # length out of range
    path[2, 2] = path[2, 3]              # not a parent link
    slots[3, 5] = 10 ** 6                # slot outside the caches
    al[4] = -1
    g, gerr = _run(kc["caches"], slots, kc["parents"], al, path)
    o, oerr = oracle.kv_compact_batch(kc["caches"], slots, kc["parents"], al, path)
    assert list(gerr) == list(oerr) == [0] + [oracle.ERR_BAD_TREE] * 4 + [0]
    assert np.array_equal(g, o)


def test_benchmark_configuration():
    kc = synth.kv_compact_case(seed=0)  # 160 caches x 976 slots x 2048 B, deepest paths (6)
    g, gerr = _run(kc["caches"], kc["slots"], kc["parents"], kc["accept_len"], kc["path"])
    o, oerr = oracle.kv_compact_batch(kc["caches"], kc["slots"], kc["parents"], kc["accept_len"], kc["path"])
    assert (gerr == 0).all() and (oerr == 0).all()
    assert np.array_equal(g, o)


def test_after_greedy_tree_verification():
    """spec_verify_tree_greedy's path feeds spec_kv_compact on the device: the request's first
    accept_len + 1 slots then hold the accepted nodes' rows in order."""
    ti = synth.tree_greedy(seed=1, B=8, V=20000, path_boost=40.0)
    g = binding.spec_verify_tree_greedy(parity.to_device(ti.target, ti.dtype), parity.i32(ti.node_tokens),
                                        parity.i32(ti.parents))
    N1 = ti.N + 1
    slots = (np.arange(ti.B)[:, None] * N1 + np.arange(N1)[None, :]).astype(np.int32)
    rows = np.arange(ti.B * N1, dtype=np.int64)
    cache = torch.from_numpy((rows[:, None] * 16 + np.arange(16)[None, :]).astype(np.uint8)).cuda()
    err = binding.spec_kv_compact([cache], parity.i32(slots), parity.i32(ti.parents), g["accept_len"],
                                  g["path_nodes"])
    torch.cuda.synchronize()
    c = cache.cpu().numpy()
    L, P = g["accept_len"].cpu().numpy(), g["path_nodes"].cpu().numpy()
    assert (err.cpu().numpy() == 0).all() and L.min() >= 1
    for b in range(ti.B):
        for j in range(L[b] + 1):
            want = (rows[b * N1 + P[b, j]] * 16 + np.arange(16)).astype(np.uint8)
            assert np.array_equal(c[b * N1 + j], want), (b, j)


def test_stream_order_around_each_call():
    """The call may be placed on the SMs while the previous kernel in the stream drains, but it
    must see all of that kernel's writes, and the next kernel must see all of its own.  A copy
    kernel refills the caches before each call and a clone reads them after it, 20 times on one
    stream, then the same sequence as a replayed CUDA graph; every result equals the oracle's."""
    kc = synth.kv_compact_case(seed=5, B=16, caches=8, row_bytes=2048)
    rng = np.random.default_rng(11)
    sets = [rng.integers(0, 256, kc["caches"].shape, dtype=np.uint8) for _ in range(4)]
    want = [oracle.kv_compact_batch(s, kc["slots"], kc["parents"], kc["accept_len"], kc["path"])[0] for s in sets]
    dev_sets = [torch.from_numpy(s).cuda() for s in sets]
    slots, parents = parity.i32(kc["slots"]), parity.i32(kc["parents"])
    al, path = parity.i32(kc["accept_len"]), parity.i32(kc["path"])
    cache = torch.empty_like(dev_sets[0])
    views = [cache[i] for i in range(cache.shape[0])]
    outs = []
    for it in range(20):
        cache.copy_(dev_sets[it % 4])
        binding.spec_kv_compact(views, slots, parents, al, path)
        outs.append(cache.clone())
    torch.cuda.synchronize()
    for it, o in enumerate(outs):
        assert np.array_equal(o.cpu().numpy(), want[it % 4]), it

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    gouts = [torch.empty_like(cache) for _ in range(4)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        binding.spec_kv_compact(views, slots, parents, al, path)  # warm-up outside the capture
        with torch.cuda.graph(graph, stream=side):
            for k in range(4):
                cache.copy_(dev_sets[k])
                binding.spec_kv_compact(views, slots, parents, al, path)
                gouts[k].copy_(cache)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        for g in gouts:
            g.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for k in range(4):
            assert np.array_equal(gouts[k].cpu().numpy(), want[k]), k


def test_limits():
    """The largest call shapes: SPEC_MAX_KV_CACHES caches and trees of SPEC_MAX_WALK_NODES nodes
    with paths of 511 and 512 moves (the move list in many batches); then 65535 requests (the
    grid's largest y extent), each moving one row."""
    N1, C = binding.MAX_WALK_NODES, binding.MAX_KV_CACHES
    par = np.array([-1, 0] + [i - 2 for i in range(2, N1)], np.int32)  # two interleaved chains
    parents = np.stack([par, par])
    path = np.full((2, N1), -1, np.int32)
    for b, last in enumerate((N1 - 2, N1 - 1)):
        chain = [last]
        while chain[-1] != 0:
            chain.append(int(par[chain[-1]]))
        chain = chain[::-1]
        path[b, : len(chain)] = chain
    al = (path >= 0).sum(1).astype(np.int32) - 1
    assert list(al) == [511, 512]
    rng = np.random.default_rng(3)
    S = 2 * N1 + 5
    slots = rng.permutation(S)[: 2 * N1].reshape(2, N1).astype(np.int32)
    caches = rng.integers(0, 256, (C, S, 16), dtype=np.uint8)
    g, gerr = _run(caches, slots, parents, al, path)
    o, oerr = oracle.kv_compact_batch(caches, slots, parents, al, path)
    assert (gerr == 0).all() and (oerr == 0).all()
    assert np.array_equal(g, o)

    B = 65535
    parents = np.tile(np.array([-1, 0, 0], np.int32), (B, 1))
    path = np.tile(np.array([0, 2, -1], np.int32), (B, 1))
    al = np.ones(B, np.int32)
    slots = (np.arange(B)[:, None] * 3 + np.arange(3)[None, :]).astype(np.int32)
    caches = rng.integers(0, 256, (1, 3 * B, 16), dtype=np.uint8)
    g, gerr = _run(caches, slots, parents, al, path)
    o, oerr = oracle.kv_compact_batch(caches, slots, parents, al, path)
    assert (gerr == 0).all() and (oerr == 0).all()
    assert np.array_equal(g, o)
    assert np.array_equal(g[0, 1::3], caches[0, 2::3])  # every request's node 2 moved to its slot 1
