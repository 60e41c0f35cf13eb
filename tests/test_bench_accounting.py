"""The bytes and rows bench.py credits to each workload (CPU only): the walk's bytes follow its own
path, the KV compaction counts only the rows that move, and every workload's algorithmic bytes
cover its logits (or rows) once."""

import os
import sys
from types import SimpleNamespace

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decoding_verification_82_gb300 import synth  # noqa: E402


class _T:  # the few tensor methods walk_read_bytes uses
    def __init__(self, a):
        self.a = np.asarray(a)

    def cpu(self):
        return self

    def numpy(self):
        return self.a


def test_walk_read_bytes_follows_the_path():
    w = dict(bench.WORKLOADS["tree_sample"])
    B, N1, V = w["B"], w["N"] + 1, w["V"]
    par = synth.eagle_tree_parents()
    L = np.zeros(B, np.int32)
    path = np.full((B, N1), -1, np.int32)
    path[:, 0] = 0
    L[1] = 2
    path[1, 1:3] = [1, 11]  # root -> node 1 -> node 11 (both have children)
    case = SimpleNamespace(out={"accept_len": _T(L), "path_nodes": _T(path)},
                           parents=_T(np.broadcast_to(par, (B, N1))))
    got = bench.walk_read_bytes(w, case)
    # every request visits the root (target + draft rows); request 1 also nodes 1 and 11
    rows = 2 * B + 4
    small = B * N1 * 4 * 2 + B * N1 * 4 + B * 4
    out = B * 4 + 2 * B * N1 * 4 + B * 4 + B * 4
    assert got == rows * V * 2 + small + out
    wg = dict(bench.WORKLOADS["tree_walk_greedy"])  # greedy: target rows only
    assert bench.walk_read_bytes(wg, case) == (B + 2) * V * 2 + B * N1 * 4 * 2 + out


def test_kv_moves_skip_rows_already_in_place():
    kc = synth.kv_compact_case(seed=0, B=16, caches=1, row_bytes=16)
    # the benchmark tree's deepest paths start at node 1, which is already in position 1
    assert (kc["path"][:, 1] == 1).all() and bench.kv_moves(kc) == 5.0
    w = dict(bench.WORKLOADS["kv_compact"], moves=5.0)
    assert bench.rows_per_request(w) == 160 * 5
    assert bench.algorithmic_bytes(w) == 2 * 16 * 800 * 2048 + 4 * 16 * 61 * 4 + 16 * 4


def test_algorithmic_bytes_cover_the_logits_once():
    for name, w in bench.WORKLOADS.items():
        w = dict(w, moves=5.0)
        if w["kind"] == "kv":
            continue
        es = 4 if w["dtype"] == "f32" else 2
        logits = w["B"] * bench.rows_per_request(w) * w["V"] * es
        extra = bench.algorithmic_bytes(w) - logits
        assert 0 < extra < 0.05 * logits, name
    # a sampled walk's rows: the 61 target rows and the draft rows of the 20 nodes with children
    assert bench.rows_per_request(bench.WORKLOADS["tree_sample"]) == 61 + 20
    assert bench.rows_per_request(bench.WORKLOADS["tree_walk_greedy"]) == 61
    assert bench.launches_per_step(bench.WORKLOADS["ngram_pipeline"]) == 2


def test_gpus_flag_never_silently_times_one_gpu(monkeypatch):
    """`--gpus N` that disagrees with the launcher's WORLD_SIZE fails; without a launcher, N > 1
    starts N ranks through torch's launcher (127.0.0.1) instead of timing one GPU."""
    import subprocess
    import sys

    env = dict(os.environ, WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2"], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 2 and "--gpus 2" in r.stderr
    calls = []
    monkeypatch.setattr(bench.subprocess, "call", lambda cmd: calls.append(cmd) or 0)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "4", "--steps", "10"])
    with pytest.raises(SystemExit) as ex:
        bench.main()
    assert ex.value.code == 0
    cmd = calls[0]
    assert cmd[1:3] == ["-m", "torch.distributed.run"] and "--nproc-per-node=4" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1" and cmd[-4:] == ["--gpus", "4", "--steps", "10"]
