#!/usr/bin/env python
"""Benchmark of the speculative-decoding verification step on GB300.

One "step" is one verification call over one batch of the workload (all steps of the hot path:
softmax statistics, acceptance scan, residual / bonus draw, or the tree argmax and walk): one
kernel launch (the residual pass of draft-model chains, which re-reads the rejected pair, runs
inside it).  Default workload: chain verification with draft-model logits,
B=64, K=5, V=128256, fp32, T=1.0 (704 logits rows, 361 MB per step).

Prints ONE JSON line (rank 0).  `value` = verified logits rows per second (whole job), timed on
the device with CUDA events, inputs resident in HBM; `e2e` = the same metric through the public
API with the step's inputs copied from pinned host memory and the results read back;
`roofline` = algorithmic bytes per call over the call's mean device time (the timed region's
CUDA-event interval over its calls, which run back to back from a replayed CUDA graph of C ABI
calls), against the measured HBM copy bandwidth; `cpu_baseline` = the CPU oracle on the host
cores.

  python bench.py [--gpus N] [--steps K] [--warmup W]
                  [--workload chain_batched|tree_greedy|ngram|tree_sample|tree_walk_greedy|ngram_pipeline|
                              kv_compact]
  python bench.py --impl reference ...   (the CPU oracle as the reference arm)
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "verify rows/sec and achieved HBM GB/s (fraction of GB300 peak) at V=128256"
WORKLOADS = {
    "chain_batched": dict(kind="chain", B=64, K=5, V=128256, dtype="f32", T=1.0,
                          desc="chain verify, batched: B=64 K=5 V=128256 fp32 T=1.0, draft-model logits"),
    "tree_greedy": dict(kind="tree", B=16, N=60, V=128256, dtype="bf16",
                        desc="greedy tree verify: B=16, 61-node EAGLE-2-like tree (depth 6), V=128256 bf16"),
    "ngram": dict(kind="ngram", B=256, K=5, V=151936, dtype="bf16", T=0.8,
                  desc="n-gram prompt-lookup verify: B=256 K=5 V=151936 bf16 T=0.8, one-hot draft"),
    # tree verification by walking (reads only the visited rows)
    "tree_sample": dict(kind="walk", B=16, N=60, V=128256, dtype="bf16", T=1.0,
                        desc="stochastic tree verify by walking: B=16, 61-node EAGLE-2-like tree, V=128256 "
                             "bf16 T=1.0, target + draft logits, children drawn from the draft"),
    # prompt lookup drafting on the GPU feeding the n-gram verification (two launches a step)
    "ngram_pipeline": dict(kind="ngram_pipe", B=256, K=5, V=151936, dtype="bf16", T=0.8, L=2052,
                           desc="n-gram pipeline: GPU prompt lookup (n=4..1) over B=256 contexts of 2052 tokens, "
                                "then n-gram verify K=5 V=151936 bf16 T=0.8"),
    # accepted-path KV-cache compaction after tree verification (Llama-3.3-70B cache geometry)
    "kv_compact": dict(kind="kv", B=16, N=60, V=0, C=160, W=2048, dtype="u8",
                       desc="accepted-path KV compaction: B=16, 61-node tree, deepest accepted paths (6 tokens), "
                            "160 K/V caches (80 layers x 8 KV heads x 128 bf16) of 2048-byte rows"),
    "tree_sample_mixed": dict(kind="walk", B=16, N=60, V=128256, dtype="bf16", T=1.0,
                              temps=(0.0, 0.6, 1.0, 1.4),
                              desc="tree verify by walking, per-request temperature: B=16 requests at T = 0, 0.6, "
                                   "1.0, 1.4 (cycled), 61-node EAGLE-2-like tree, V=128256 bf16, target + draft logits"),
    "tree_walk_greedy": dict(kind="walk", B=16, N=60, V=128256, dtype="bf16", T=0.0,
                             desc="greedy tree verify by walking: B=16, 61-node EAGLE-2-like tree (depth 6), "
                                  "V=128256 bf16"),
    # per-request temperature on the streaming calls (T = 0 requests verified greedily)
    "chain_mixed": dict(kind="chain", B=64, K=5, V=128256, dtype="f32", T=1.0, temps=(0.0, 0.6, 1.0, 1.4),
                        desc="chain verify, per-request temperature: B=64 K=5 V=128256 fp32, draft-model logits, "
                             "T = 0, 0.6, 1.0, 1.4 cycled over the requests (T = 0: greedy, draft rows not read)"),
    "ngram_mixed": dict(kind="ngram", B=256, K=5, V=151936, dtype="bf16", T=0.8, temps=(0.0, 0.6, 1.0, 1.4),
                        desc="n-gram prompt-lookup verify, per-request temperature: B=256 K=5 V=151936 bf16, "
                             "one-hot draft, T = 0, 0.6, 1.0, 1.4 cycled over the requests"),
}
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # GB300's nominal HBM3e bandwidth (~8 TB/s), for context beside the measured peak
KERNEL_SOURCES = ["speculative_decoding_verification_82_gb300/csrc/verify_kernel.cuh",
                  "speculative_decoding_verification_82_gb300/csrc/verify_common.cuh",
                  "speculative_decoding_verification_82_gb300/csrc/fastdiv.h",
                  "speculative_decoding_verification_82_gb300/csrc/spec_verify_api.cu"]
KV_SOURCES = ["speculative_decoding_verification_82_gb300/csrc/kv_compact.cu"]
WALK_SOURCES = ["speculative_decoding_verification_82_gb300/csrc/tree_walk.cuh",
                "speculative_decoding_verification_82_gb300/csrc/verify_common.cuh",
                "speculative_decoding_verification_82_gb300/csrc/spec_walk.cu"]


# ----------------------------------------------------------------------------- inputs ----
def make_inputs(name: str, seed: int):
    from speculative_decoding_verification_82_gb300 import synth

    if name in ("chain_batched", "chain_mixed"):
        return synth.chain_batched(seed=seed)
    if name == "tree_greedy":
        return synth.tree_greedy(seed=seed)
    if name in ("ngram", "ngram_mixed"):
        return synth.ngram(seed=seed)
    if name == "tree_sample":
        return synth.tree_sample(seed=seed)
    if name == "tree_walk_greedy":
        return synth.tree_greedy(seed=seed)
    if name == "tree_sample_mixed":
        return synth.tree_sample(seed=seed)
    if name == "kv_compact":
        return synth.kv_compact_case(seed=seed)
    if name == "ngram_pipeline":
        ci = synth.ngram(seed=seed)
        ci.meta["ctx"], ci.meta["ctx_len"] = synth.ngram_contexts(seed=seed)
        return ci
    raise ValueError(name)


def request_temps(w: dict, B: int):
    """The per-request temperatures of a workload that has them (cycled over the requests), else None."""
    return np.resize(np.asarray(w["temps"], np.float32), B) if "temps" in w else None


def rows_per_request(w: dict) -> float:
    """Logits rows a request supplies: a walk's draft rows count for the nodes with children (the
    rows that exist as the draft's output), 20 of the 61 nodes of the benchmark tree; with
    per-request temperatures a chain request verified greedily reads its K + 1 target rows only
    (the mean over the batch)."""
    if w["kind"] == "chain" and "temps" in w:
        t = request_temps(w, w["B"])
        return float(np.mean(np.where(t == 0, w["K"] + 1, 2 * w["K"] + 1)))
    if w["kind"] == "chain":
        return 2 * w["K"] + 1
    if w["kind"] in ("ngram", "ngram_pipe"):
        return w["K"] + 1
    if w["kind"] == "kv":
        return w["C"] * w["moves"]  # rows moved per request (set from the inputs by kv_moves)
    if w["kind"] == "walk" and (w["T"] > 0 or "temps" in w):
        from speculative_decoding_verification_82_gb300 import synth

        par = synth.eagle_tree_parents()
        return par.size + int(np.unique(par[1:]).size)
    return w["N"] + 1


KV_METRIC = "KV-cache rows compacted per second (a row: one token's K or V in one layer) and achieved HBM GB/s"
KV_ORACLE_CACHES = 8  # the CPU oracle's sample moves the rows of this many of the caches


def workload_metric(w: dict) -> str:
    return KV_METRIC if w["kind"] == "kv" else METRIC


def kv_moves(inp) -> float:
    """Mean number of rows a request's compaction moves in one cache: accepted positions j whose
    node is not already in position j's slot (those are skipped).  Along the benchmark tree's
    deepest paths the first accepted node is node 1, so 5 of the 6 accepted rows move."""
    sl, pt, al = inp["slots"], inp["path"], inp["accept_len"]
    n = [sum(int(sl[b, pt[b, j]] != sl[b, j]) for j in range(1, al[b] + 1)) for b in range(len(al))]
    return float(np.mean(n))


def graph_calls(K: int) -> int:
    """Calls per captured graph: the largest divisor of K up to 50, so that whole replays time
    exactly K calls."""
    return max(d for d in range(1, min(K, 50) + 1) if K % d == 0)


def launches_per_step(w: dict) -> int:
    """Kernel launches of one step: verify_kernel (which also makes the residual pass of
    draft-model chains) or walk_kernel; the n-gram pipeline adds the lookup kernel."""
    return 2 if w["kind"] == "ngram_pipe" else 1


def algorithmic_bytes(w: dict) -> int:
    """Logits read once, the small inputs read once, the outputs written once."""
    B, V = w["B"], w["V"]
    if w["kind"] == "kv":  # every moved row read once and written once, plus the path arrays
        return 2 * B * rows_per_request(w) * w["W"] + 4 * B * (w["N"] + 1) * 4 + B * 4
    es = 4 if w["dtype"] == "f32" else 2
    logits = int(round(B * rows_per_request(w))) * V * es
    if w["kind"] in ("tree", "walk"):
        small_in = 2 * B * (w["N"] + 1) * 4
        out = B * 4 + 2 * B * (w["N"] + 1) * 4 + B * 4
    else:
        K = w["K"]
        small_in = B * K * 4 * 2 + B * 4
        out = B * 4 + B * (K + 1) * 4 + B * 4 + B * 4
        if w["kind"] == "ngram_pipe":  # contexts and lengths read, drafts written (and read back)
            small_in += B * w["L"] * 4 + B * 4 + B * K * 4
            out += B * K * 4 + 4 * B * 4
    return logits + small_in + out


def walk_read_bytes(w: dict, case) -> int:
    """Bytes a tree walk call reads for the outputs it produced: per request, the target row of
    every visited node and the draft row of every visited node with children (T > 0), plus the
    tree arrays, the uniforms and the outputs."""
    B, N1, V = w["B"], w["N"] + 1, w["V"]
    es = 4 if w["dtype"] == "f32" else 2
    L = case.out["accept_len"].cpu().numpy()
    path = case.out["path_nodes"].cpu().numpy()
    par = case.parents.cpu().numpy()
    total = 0
    for b in range(B):
        has_kids = np.zeros(N1, bool)
        has_kids[par[b, 1:]] = True
        nodes = path[b, : L[b] + 1]
        Tb = np.resize(np.asarray(w["temps"], np.float32), B)[b] if "temps" in w else w["T"]
        rows = len(nodes) + (int(has_kids[nodes].sum()) if Tb > 0 else 0)
        total += rows * V * es
    small = B * N1 * 4 * 2 + (B * N1 * 4 + B * 4 if (w["T"] > 0 or "temps" in w) else 0)
    out = B * 4 + 2 * B * N1 * 4 + B * 4 + B * 4
    return total + small + out


# ------------------------------------------------------------------------------ clocks ----
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        inside = [l for t, l in self.lines if t0 <= t <= t1]
        window = "timed region"
        if not inside:  # timed region shorter than the sampling interval: nearest samples
            inside = [l for t, l in self.lines if t0 - 0.2 <= t <= t1 + 0.2]
            window = "timed region +- 0.2 s"
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in inside:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "window": window}


# --------------------------------------------------------------------- peaks / traffic ----
def hbm_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "of measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "of fallback"


def kernel_source_hash(workload: str = "chain_batched") -> str:
    h = hashlib.sha256()
    kind = WORKLOADS[workload]["kind"]
    for rel in (WALK_SOURCES if kind == "walk" else KV_SOURCES if kind == "kv" else KERNEL_SOURCES):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per call from the committed ncu summary, if it matches the current kernels."""
    p = os.path.join(ROOT, "profiles", f"verify_{workload}.md")
    try:
        text = open(p).read()
    except OSError:
        return None
    m_b = re.search(r"traffic_bytes_per_call:\s*([0-9]+)", text)
    m_h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m_b or not m_h or m_h.group(1) != kernel_source_hash(workload):
        return None
    return int(m_b.group(1))


# -------------------------------------------------------------------------- CPU oracle ----
def oracle_run(w: dict, inp, requests, threads: int):
    import oracle

    if w["kind"] == "chain":
        return oracle.verify_chain(inp.dtype, inp.target, inp.draft, inp.B, inp.K, inp.V,
                                   float(inp.temperature), inp.draft_tokens, inp.r, inp.u,
                                   threads=threads, requests=requests, temperatures=request_temps(w, inp.B))
    if w["kind"] == "ngram":
        return oracle.verify_ngram(inp.dtype, inp.target, inp.B, inp.K, inp.V, float(inp.temperature),
                                   inp.draft_tokens, inp.r, inp.u, threads=threads, requests=requests,
                                   temperatures=request_temps(w, inp.B))
    if w["kind"] == "kv":
        b0, b1 = requests
        return oracle.kv_compact_batch(inp["caches"][:KV_ORACLE_CACHES], inp["slots"][b0:b1], inp["parents"][b0:b1],
                                       inp["accept_len"][b0:b1], inp["path"][b0:b1])
    if w["kind"] == "ngram_pipe":
        b0, b1 = requests
        d = oracle.ngram_draft_batch(inp.meta["ctx"][b0:b1], inp.meta["ctx_len"][b0:b1], inp.K)
        x = inp.draft_tokens.copy()
        x[b0:b1] = d["draft"]
        return oracle.verify_ngram(inp.dtype, inp.target, inp.B, inp.K, inp.V, float(inp.temperature),
                                   x, inp.r, inp.u, threads=threads, requests=requests)
    if w["kind"] == "walk":
        T = float(w["T"])
        temps = np.resize(np.asarray(w["temps"], np.float32), inp.B) if "temps" in w else None
        sampled = T > 0 or temps is not None
        return oracle.verify_tree_sample(inp.dtype, inp.target, inp.draft if sampled else None, inp.B,
                                         inp.N, inp.V, T, inp.node_tokens, inp.parents,
                                         inp.r if sampled else None, inp.u if sampled else None,
                                         threads=threads, requests=requests, temperatures=temps)
    return oracle.verify_tree_greedy(inp.dtype, inp.target, inp.B, inp.N, inp.V, inp.node_tokens,
                                     inp.parents, threads=threads, requests=requests)


def oracle_timed(w: dict, inp, n_req: int, threads: int) -> float:
    """Wall time of the oracle over requests [0, n_req), requests split across threads (ctypes
    releases the GIL, so each thread runs on its own core)."""
    import oracle

    rngs = oracle._ranges(n_req, threads)
    t0 = time.perf_counter()
    ts = [threading.Thread(target=oracle_run, args=(w, inp, rg, 1)) for rg in rngs]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    return time.perf_counter() - t0


def cpu_baseline(w: dict, inp, min_wall: float = 1.0) -> dict:
    cores = os.cpu_count() or 1
    n_req = w["B"]
    threads = min(cores, n_req)
    reps, wall = 0, 0.0
    while wall < min_wall or reps < 2:
        wall += oracle_timed(w, inp, n_req, threads)
        reps += 1
    rows = reps * n_req * rows_per_request(w)
    if w["kind"] == "kv":
        rows = rows * KV_ORACLE_CACHES / w["C"]
    note = f", the rows of {KV_ORACLE_CACHES} of the {w['C']} caches" if w["kind"] == "kv" else ""
    return {"value": rows / wall, "unit": "rows/s", "cores": threads, "kind": "oracle",
            "sample": f"all {n_req} requests of the workload ({rows / reps:g} rows{note}), "
                      f"{reps} repetitions, requests split over {threads} threads, {wall:.2f} s wall"}


# ------------------------------------------------------------------------ GPU arm ----
def dist_setup():
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seeds(rank: int, n_sets: int) -> list[int]:
    """Input seeds of one rank: each rank verifies its own requests (the path shards by request)."""
    return [1000 * rank + s for s in range(n_sets)]


def job_rows_per_s(world: int, rows_per_step: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job throughput: every rank processed `rows_per_step` rows per step; the slowest
    rank's time (max over ranks) bounds the job."""
    return world * rows_per_step * steps / (elapsed_ms / 1e3)


class DeviceCase:
    """One input set (on the device, or in pinned host memory) plus preallocated outputs;
    `call()` is one step through the public binding."""

    def __init__(self, w, inp, dev, workspace, host_pinned: bool = False):
        import torch

        from speculative_decoding_verification_82_gb300 import binding

        self.w, self.binding = w, binding
        tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "u8": torch.uint8}[w["dtype"]]

        def tens(a, dt=None):
            a = np.ascontiguousarray(a)
            t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if dt == torch.bfloat16 else torch.from_numpy(a)
            return t.pin_memory() if host_pinned else t.to(dev)

        B = w["B"]
        self.draft = None
        if w["kind"] == "kv":
            self.cache_all = tens(inp["caches"])
            self.caches = [self.cache_all[i] for i in range(w["C"])]
            self.slots, self.parents = tens(inp["slots"]), tens(inp["parents"])
            self.al, self.path = tens(inp["accept_len"]), tens(inp["path"])
            self.target = self.cache_all
            shapes = dict(err_flags=(B,))
        else:
            self.target = tens(inp.target, tdt)
        if w["kind"] == "kv":
            pass  # set above
        elif w["kind"] == "tree":
            self.tokens, self.parents = tens(inp.node_tokens), tens(inp.parents)
            N1 = w["N"] + 1
            shapes = dict(accept_len=(B,), path_nodes=(B, N1), out_tokens=(B, N1), err_flags=(B,))
        elif w["kind"] == "walk":
            self.T = float(w["T"])
            self.tokens, self.parents = tens(inp.node_tokens), tens(inp.parents)
            if "temps" in w:
                self.temps = tens(np.resize(np.asarray(w["temps"], np.float32), B))
            stoch = self.T > 0 or "temps" in w
            self.draft = tens(inp.draft, tdt) if stoch else None
            self.r = tens(inp.r) if stoch else None
            self.u = tens(inp.u) if stoch else None
            N1 = w["N"] + 1
            shapes = dict(accept_len=(B,), path_nodes=(B, N1), out_tokens=(B, N1), residual_mass=(B,),
                          err_flags=(B,))
        else:
            self.draft = tens(inp.draft, tdt) if w["kind"] == "chain" else None
            self.x, self.r, self.u = tens(inp.draft_tokens), tens(inp.r), tens(inp.u)
            if "temps" in w:
                self.temps = tens(request_temps(w, B))
            if w["kind"] == "ngram_pipe":  # the drafts come from the lookup kernel every step
                self.ctx, self.ctx_len = tens(inp.meta["ctx"]), tens(inp.meta["ctx_len"])
                dshape = dict(draft_len=(B,), match_n=(B,), match_end=(B,), err_draft=(B,))
                self.dout = {k: (torch.empty(v, dtype=torch.int32).pin_memory() if host_pinned
                                 else torch.empty(v, dtype=torch.int32, device=dev)) for k, v in dshape.items()}
            self.T = float(inp.temperature)
            K1 = w["K"] + 1
            shapes = dict(num_accepted=(B,), out_tokens=(B, K1), residual_mass=(B,), err_flags=(B,))
        fdt = {"residual_mass": torch.float32}
        if host_pinned:
            self.out = {k: torch.empty(s, dtype=fdt.get(k, torch.int32)).pin_memory() for k, s in shapes.items()}
        else:
            self.out = {k: torch.empty(s, dtype=fdt.get(k, torch.int32), device=dev) for k, s in shapes.items()}
        self.ws = workspace

    def inputs(self):
        if self.w["kind"] == "tree":
            return [self.target, self.tokens, self.parents]
        if self.w["kind"] == "kv":
            return [self.cache_all, self.slots, self.parents, self.al, self.path]
        if self.w["kind"] == "walk":
            return [t for t in (self.target, self.draft, self.tokens, self.parents, self.r, self.u,
                                getattr(self, "temps", None)) if t is not None]
        if self.w["kind"] == "ngram_pipe":
            return [self.target, self.ctx, self.ctx_len, self.r, self.u]
        return [t for t in (self.target, self.draft, self.x, self.r, self.u, getattr(self, "temps", None))
                if t is not None]

    def abi_args(self):
        """Arguments of the C ABI call itself (device pointers, sizes, the current stream), built once
        so that the device-timed loop measures the library call, not Python argument handling."""
        import ctypes

        import torch

        P = ctypes.c_void_p
        ptr = lambda t: P(t.data_ptr()) if t is not None else None  # noqa: E731
        if self.w["kind"] == "kv":
            stream = P(torch.cuda.current_stream().cuda_stream)
            self._arr = (P * len(self.caches))(*[c.data_ptr() for c in self.caches])
            return [("spec_kv_compact", (self._arr, len(self.caches), self.caches[0].shape[0], self.w["W"],
                                         self.w["B"], self.w["N"], ptr(self.slots), ptr(self.parents),
                                         ptr(self.al), ptr(self.path), ptr(self.out["err_flags"]), stream))]
        dt = self.binding.DTYPE_CODE[self.target.dtype]
        stream = P(torch.cuda.current_stream().cuda_stream)
        o = self.out
        B = self.w["B"]
        if self.w["kind"] == "walk":
            return [("spec_verify_tree_walk",
                    (ptr(self.target), ptr(self.draft), dt, B, self.w["N"], self.w["V"], ctypes.c_float(self.T),
                     ptr(getattr(self, "temps", None)), ptr(self.tokens), ptr(self.parents), ptr(self.r), ptr(self.u), ptr(o["accept_len"]),
                     ptr(o["path_nodes"]), ptr(o["out_tokens"]), ptr(o["residual_mass"]), ptr(o["err_flags"]),
                     None, stream))]
        ws, nbytes = ptr(self.ws), self.ws.numel()
        if self.w["kind"] == "tree":
            return [("spec_verify_tree_greedy",
                     (ptr(self.target), dt, B, self.w["N"], self.w["V"], ptr(self.tokens), ptr(self.parents),
                      ptr(o["accept_len"]), ptr(o["path_nodes"]), ptr(o["out_tokens"]), ptr(o["err_flags"]), None,
                      ws, nbytes, stream))]
        K, V = self.w["K"], self.w["V"]
        tail = (ptr(o["num_accepted"]), ptr(o["out_tokens"]), ptr(o["residual_mass"]), ptr(o["err_flags"]),
                None, None, None, None)
        verify = ("spec_verify_ngram", (ptr(self.target), dt, B, K, V, ctypes.c_float(self.T),
                                        ptr(getattr(self, "temps", None)), ptr(self.x),
                                        ptr(self.r), ptr(self.u), *tail, ws, nbytes, stream))
        if self.w["kind"] == "ngram_pipe":
            d = self.dout
            return [("spec_ngram_draft", (ptr(self.ctx), ptr(self.ctx_len), B, self.ctx.shape[1], 4, 1, K,
                                          ptr(self.x), ptr(d["draft_len"]), ptr(d["match_n"]), ptr(d["match_end"]),
                                          ptr(d["err_draft"]), stream)), verify]
        if self.w["kind"] == "ngram":
            return [verify]
        return [("spec_verify_chain", (ptr(self.target), ptr(self.draft), dt, B, K, V, ctypes.c_float(self.T),
                                       ptr(getattr(self, "temps", None)),
                                       ptr(self.x), ptr(self.r), ptr(self.u), *tail, None, ws, nbytes, stream))]

    def call(self):
        b = self.binding
        if self.w["kind"] == "kv":
            return {"err_flags": b.spec_kv_compact(self.caches, self.slots, self.parents, self.al, self.path,
                                                   err_flags=self.out["err_flags"])}
        if self.w["kind"] == "walk":
            return b.spec_verify_tree_walk(self.target, self.draft, self.tokens, self.parents, self.r, self.u,
                                           self.T, out=self.out, temperatures=getattr(self, "temps", None))
        if self.w["kind"] == "tree":
            return b.spec_verify_tree_greedy(self.target, self.tokens, self.parents, workspace=self.ws, out=self.out)
        if self.w["kind"] == "ngram_pipe":
            d = b.spec_ngram_draft(self.ctx, self.ctx_len, self.w["K"],
                                   out=dict(draft_tokens=self.x, draft_len=self.dout["draft_len"],
                                            match_n=self.dout["match_n"], match_end=self.dout["match_end"],
                                            err_flags=self.dout["err_draft"]))
            return b.spec_verify_ngram(self.target, d["draft_tokens"], self.r, self.u, self.T, workspace=self.ws,
                                       out=self.out)
        tt = getattr(self, "temps", None)
        if self.w["kind"] == "ngram":
            return b.spec_verify_ngram(self.target, self.x, self.r, self.u, self.T, workspace=self.ws, out=self.out,
                                       temperatures=tt)
        return b.spec_verify_chain(self.target, self.draft, self.x, self.r, self.u, self.T, workspace=self.ws,
                                   out=self.out, temperatures=tt)


def _e2e_step(dev_case: DeviceCase, host_case: DeviceCase):
    for d, h in zip(dev_case.inputs(), host_case.inputs()):
        d.copy_(h, non_blocking=True)
    dev_case.call()
    for k, t in dev_case.out.items():
        host_case.out[k].copy_(t, non_blocking=True)


def parity_summary(w: dict, name: str, inp, dev, ws) -> dict:
    """One call of the workload on its seed-0 inputs, outside the timed region, checked against the
    oracle on the same inputs with the parity rule of the tests: counts of the requests that match
    exactly, of the oracle's flagged-tie set (strict: within 1e-6; widened-only: within the 1e-6 / S
    band of a residual, not 1e-6), of flagged requests that took an admissible alternative, and of
    failures (0 is the bar)."""
    import torch

    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import parity

    from speculative_decoding_verification_82_gb300 import binding

    kind = w["kind"]
    if kind == "kv":
        import oracle

        caches = torch.from_numpy(np.ascontiguousarray(inp["caches"][:KV_ORACLE_CACHES])).to(dev)
        ii = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)  # noqa: E731
        e = binding.spec_kv_compact([caches[i] for i in range(caches.shape[0])], ii(inp["slots"]),
                                    ii(inp["parents"]), ii(inp["accept_len"]), ii(inp["path"]))
        torch.cuda.synchronize()
        ref, err = oracle.kv_compact_batch(inp["caches"][:KV_ORACLE_CACHES], inp["slots"], inp["parents"],
                                           inp["accept_len"], inp["path"])
        same = bool(np.array_equal(caches.cpu().numpy(), ref)) and bool(np.array_equal(e.cpu().numpy(), err))
        return {"seed": 0, "requests": int(w["B"]), "caches_checked": KV_ORACLE_CACHES,
                "bytes_exact": same, "failures": 0 if same else 1}
    threads = os.cpu_count() or 1
    if kind == "tree":
        g = parity.run_gpu_tree(inp, workspace=ws)
        o = parity.run_oracle_tree(inp, threads=threads)
        fails = sum(int(not np.array_equal(g[a][b], o[c][b])) for b in range(inp.B)
                    for a, c in (("accept_len", "accept_len"), ("path_nodes", "path"), ("out_tokens", "out_tokens"),
                                 ("node_argmax", "amax"), ("err_flags", "err")))
        return {"seed": 0, "requests": int(inp.B), "exact": int(inp.B) if not fails else None, "failures": fails,
                "rule": "bit-exact (argmax, path, tokens, error bits)"}
    if kind == "walk":
        temps = np.resize(np.asarray(w["temps"], np.float32), inp.B) if "temps" in w else None
        g = parity.run_gpu_walk(inp, float(w["T"]), temperatures=temps)
        o = parity.run_oracle_walk(inp, float(w["T"]), threads=threads, temperatures=temps)
        st = parity.check_walk(g, o, inp)
    else:
        ngram = kind in ("ngram", "ngram_pipe")
        temps = request_temps(w, inp.B)
        g = parity.run_gpu_chain(inp, ngram=ngram, workspace=ws, diag=False, temperatures=temps)
        o = parity.run_oracle_chain(inp, ngram=ngram, threads=threads, temperatures=temps)
        st = parity.check_chain(g, o, inp)
    out = {k: st[k] for k in ("requests", "errors", "flagged_strict", "flagged_wide_only",
                              "admissible_deviations")}
    out["exact"] = st["requests"] - st["admissible_deviations"] - len(st["failures"])
    out["failures"] = len(st["failures"])
    out["seed"] = 0
    out["rule"] = ("bit-exact outside the flagged-tie set; flagged requests: an admissible outcome "
                   "(the other decision of a tied accept test, or a positive-weight token whose CDF "
                   "interval comes within the tie band of u)")
    return out


def measure(args, name: str, w: dict, rank: int, world: int, local: int, primary: bool) -> dict:
    """Times K steps of workload `name` (a replayed CUDA graph of C ABI calls) and returns its JSON
    fields; the primary workload also gets the end-to-end figure, the CPU oracle and the parity
    summary."""
    import torch

    from speculative_decoding_verification_82_gb300 import binding

    dev = torch.device("cuda", local)
    # alternate input sets; each is larger than L2 as well, except the KV compaction's 63 MB of moved
    # rows per step, which takes four sets (252 MB touched per round, about twice L2)
    n_sets = 4 if w["kind"] == "kv" else 2
    inputs = [make_inputs(name, seed=s) for s in rank_seeds(rank, n_sets)]
    if w["kind"] == "kv":
        w["moves"] = float(np.mean([kv_moves(inp) for inp in inputs]))
    rows_req = rows_per_request(w)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "u8": torch.uint8}[w["dtype"]]
    ws_rows = 2 * w["K"] + 1 if w["kind"] == "chain" else int(rows_req)  # (any request may read its draft rows)
    ws = None if w["kind"] in ("walk", "kv") else binding.make_workspace(w["B"], ws_rows, w["V"], tdt, dev)
    cases = [DeviceCase(w, inp, dev, ws) for inp in inputs]
    stream = torch.cuda.current_stream(dev)

    for i in range(args.warmup):
        cases[i % n_sets].call()
    torch.cuda.synchronize()
    barrier(world)
    # the timed loop calls the C ABI directly with prepared arguments (the binding's checks cost
    # host time that would otherwise show up as gaps between calls on the device)
    lib = binding.library()
    abi = []
    for c in cases:
        abi.append([(getattr(lib, fn_name), a) for fn_name, a in c.abi_args()])
    visited = []
    for c, calls in zip(cases, abi):
        for fn, a in calls:
            st = fn(*a)
            if st != binding.SPEC_OK:
                raise RuntimeError(f"C ABI call failed: {lib.spec_status_string(st).decode()}")
        if w["kind"] == "walk":
            torch.cuda.synchronize()
            visited.append(walk_read_bytes(w, c))
    torch.cuda.synchronize()

    K = args.steps
    # The timed steps run from a CUDA graph of C ABI calls (alternating the input sets), captured
    # once and replayed, so that the host's rate of issuing calls cannot leave the device idle
    # between them.  Each replayed call is a full call: its tag comes from the workspace's epoch.
    per_graph = graph_calls(K)
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        gabi = []
        for c in cases:  # the calls' stream argument: the capturing stream
            gabi.append([(getattr(lib, fn_name), a) for fn_name, a in c.abi_args()])
        status = 0
        for i in range(per_graph):
            for fn, a in gabi[i % n_sets]:
                status |= fn(*a)
    if status != binding.SPEC_OK:
        raise RuntimeError("a captured C ABI call failed")
    graph.replay()  # one untimed replay
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.15)
    torch.cuda.synchronize()
    barrier(world)
    t_host0 = time.perf_counter()
    start.record(stream)
    for _ in range(K // per_graph):
        graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.perf_counter()
    barrier(world)
    clk = clocks.stop(t_host0, t_host1)
    elapsed_ms = max_over_ranks(start.elapsed_time(end), world)
    mean_call_ms = start.elapsed_time(end) / K  # device time per call, back to back
    del graph

    rows_step = int(round(w["B"] * rows_req))
    value = job_rows_per_s(world, rows_step, K, elapsed_ms)
    alg_bytes = algorithmic_bytes(w)
    read_bytes = float(np.mean(visited)) if visited else float(alg_bytes)
    achieved = read_bytes / (mean_call_ms / 1e3) / 1e9
    peak, peak_src = hbm_peak()
    res = {
        "value": value, "ms_per_step": elapsed_ms / K, "steps": K,
        "config": {"workload": w["desc"], "B": w["B"], "V": w["V"],
                   **({"K": w["K"]} if "K" in w else {"N": w["N"]}),
                   "rows_per_step": rows_step, "requests_per_s": value / rows_req,
                   "l2": f"{alg_bytes / 2**20:.0f} MiB touched per step, {n_sets} input sets alternated "
                         f"({n_sets * alg_bytes / 2**20:.0f} MiB per round; L2 129 MiB)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_src,
                     "frac_of_nominal_8TBs": achieved / NOMINAL_HBM_GBS,
                     "traffic": profiled_traffic(name), "algorithmic_bytes_per_call": read_bytes,
                     "mean_call_us": mean_call_ms * 1e3,
                     "kernel": (f"verify_kernel<ngram,{w['dtype']}> after ngram_draft_kernel (two launches a step)"
                                if w["kind"] == "ngram_pipe" else
                                f"verify_kernel<{w['kind']},{w['dtype']}> (one launch per call)")},
        "gpu_launches": K * launches_per_step(w),
        "clocks": clk,
    }
    if w["kind"] == "kv":
        res["roofline"]["kernel"] = "kv_compact_kernel (one launch per call)"
        res["config"]["rows"] = (f"moved rows ({w['moves']:g} per request and cache: accepted positions whose node is "
                                 f"not already in place) x 2048 bytes, read and written once")
    if w["kind"] == "walk":
        res["roofline"].update(
            kernel=("walk_kernel (one launch per call): 6-CTA clusters with 48 tokens a thread when they take "
                    "the batch in fewer waves than 8-CTA clusters with 32 (greedy: p in registers; one "
                    "temperature: p and q in shared memory), else 8-CTA clusters; per-request temperatures: "
                    "8-CTA clusters"),
            algorithmic_bytes_note="acceptance-aware: the rows the walk reads (visited nodes' target rows, and "
                                   "draft rows of visited nodes with children), mean over the input sets",
            all_rows_bytes_per_call=alg_bytes,
            all_rows_equivalent_GBs=alg_bytes / (mean_call_ms / 1e3) / 1e9,
            note="latency-bound: one row pair per tree level, read by one cluster per request; the "
                 "all-rows figure is the bandwidth a pass over every row would need to match this time")
    if primary:
        # ---- end to end through the public API: pinned host -> device, call, results -> host ----
        host = [DeviceCase(w, inp, dev, ws, host_pinned=True) for inp in inputs]
        e2e_steps = max(3, min(K, args.e2e_steps))
        h2d = sum(t.numel() * t.element_size() for t in host[0].inputs())
        d2h = sum(t.numel() * t.element_size() for t in host[0].out.values())
        for i in range(2):
            _e2e_step(cases[i % n_sets], host[i % n_sets])
        torch.cuda.synchronize()
        barrier(world)
        e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_s.record(stream)
        for i in range(e2e_steps):
            _e2e_step(cases[i % n_sets], host[i % n_sets])
        e_e.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e_s.elapsed_time(e_e), world)
        res["e2e"] = {"value": world * rows_step * e2e_steps / (e2e_ms / 1e3), "unit": "rows/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                      "ms_per_step": e2e_ms / e2e_steps}
        del host
    if rank == 0 and not args.no_cpu_baseline:
        if primary:
            res["cpu_baseline"] = cpu_baseline(w, inputs[0])
        if world == 1:  # the seed-0 inputs are rank 0's first set
            res["parity"] = parity_summary(w, name, inputs[0], dev, ws)
    del cases
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


# workloads the default run also times, reported under "secondary" (same process, same GPU)
SECONDARY = ("tree_greedy", "ngram")


def run_gpu(args, w) -> None:
    import torch

    from speculative_decoding_verification_82_gb300 import binding

    rank, world, local = dist_setup()
    torch.cuda.set_device(local)
    binding.library()  # fail loudly if the CUDA library is missing
    res = measure(args, args.workload, w, rank, world, local, primary=True)
    secondary = {}
    if args.workload == "chain_batched" and not args.no_secondary:
        for name in SECONDARY:
            sw = WORKLOADS[name]
            r2 = measure(args, name, sw, rank, world, local, primary=False)
            secondary[name] = {"workload": sw["desc"], "value": r2["value"], "unit": "rows/s",
                               "ms_per_step": r2["ms_per_step"], "roofline": r2["roofline"],
                               "clocks": r2["clocks"], "gpu_launches": r2["gpu_launches"],
                               **({"parity": r2["parity"]} if "parity" in r2 else {})}
    if rank != 0:
        return
    line = {
        "metric": workload_metric(w),
        "value": res["value"],
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": res["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w["dtype"],
        "data": "synthetic (seeded Philox; logits, tokens and uniforms per the workload recipe)",
        "config": res["config"],
        "roofline": res["roofline"],
        "e2e": res["e2e"],
        "gpu_launches": res["gpu_launches"] + sum(v["gpu_launches"] for v in secondary.values()),
        "gpu_launches_primary": res["gpu_launches"],
        "clocks": res["clocks"],
    }
    for k in ("cpu_baseline", "parity"):
        if k in res:
            line[k] = res[k]
    if secondary:
        line["secondary"] = secondary
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ reference arm ----
def run_reference(args, w) -> None:
    """The CPU oracle as the reference arm (the pages give no implementation to install)."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    inp = make_inputs(args.workload, seed=0)
    if w["kind"] == "kv":
        w["moves"] = kv_moves(inp)
    cores = os.cpu_count() or 1
    t_one = oracle_timed(w, inp, 1, 1)
    budget = 150.0 / max(1, args.steps + args.warmup)  # keep the whole run within a few minutes
    n_req = int(max(1, min(w["B"], cores * budget / max(t_one, 1e-6))))
    threads = min(cores, n_req)
    for _ in range(args.warmup):
        oracle_timed(w, inp, n_req, threads)
    t = 0.0
    for _ in range(args.steps):
        t += oracle_timed(w, inp, n_req, threads)
    # the KV compaction's oracle sample moves the rows of KV_ORACLE_CACHES of the caches
    scale = KV_ORACLE_CACHES / w["C"] if w["kind"] == "kv" else 1
    sample_note = f" of {KV_ORACLE_CACHES} of the {w['C']} caches" if w["kind"] == "kv" else ""
    value = args.steps * n_req * rows_per_request(w) * scale / t
    line = {
        "impl": "reference",
        "metric": workload_metric(w),
        "value": value, "unit": "rows/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w["dtype"],
        "data": "synthetic (seeded Philox)",
        "config": {"workload": w["desc"], "B": w["B"], "V": w["V"],
                   "rows_per_step": n_req * rows_per_request(w) * scale},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n_req} request(s) of the workload per step "
                                   f"({n_req * rows_per_request(w) * scale:g} rows{sample_note}), "
                                   f"split over {threads} threads"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def free_port() -> int:
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def spawn_ranks(n: int) -> int:
    """`--gpus N` without a launcher: starts N local ranks (one per GPU) through torch's launcher on
    127.0.0.1, with the same arguments; rank 0 prints the line.  Returns the launcher's status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.abspath(__file__),
           *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="chain_batched", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="time only the chosen workload (the default run also times tree_greedy and ngram)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    launched = os.environ.get("WORLD_SIZE")
    if launched is None and args.gpus > 1:
        sys.exit(spawn_ranks(args.gpus))
    if int(launched or "1") != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but the launcher started {launched} rank(s)", file=sys.stderr)
        sys.exit(2)
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
