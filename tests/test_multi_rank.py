"""The multi-rank path of bench.py on the CPU: two `gloo` ranks (no GPU needed).

Each rank verifies its own requests (different seeds), ranks exchange nothing on the data path,
and the job's time is the maximum over ranks; these tests run that logic in two processes."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench

    r, w, local = bench.dist_setup()
    try:
        assert (r, w, local) == (rank, world, rank)
        assert dist.get_backend() == "gloo"
        bench.barrier(w)
        # the job time is the slowest rank's
        t = bench.max_over_ranks(10.0 + rank, w)
        seeds = bench.rank_seeds(r, 2)
        all_seeds = [None] * w
        dist.all_gather_object(all_seeds, seeds)
        value = bench.job_rows_per_s(w, rows_per_step=704, steps=100, elapsed_ms=t)
        out.put((rank, t, all_seeds, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_by_request_and_take_the_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for rank, t, all_seeds, value in res:
        assert t == 11.0  # max over ranks
        flat = [s for ss in all_seeds for s in ss]
        assert len(set(flat)) == len(flat)  # every rank has its own inputs
        assert value == pytest.approx(world * 704 * 100 / 0.011)


def test_single_rank_needs_no_process_group():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.rank_seeds(0, 2) == [0, 1] and bench.rank_seeds(1, 2) == [1000, 1001]
    assert bench.job_rows_per_s(1, 704, 2000, 1000.0) == 704 * 2000
    # calls per captured graph: a divisor of the step count, so whole replays time exactly K calls
    for K in (1, 2, 3, 7, 97, 100, 2000, 2001):
        g = bench.graph_calls(K)
        assert 1 <= g <= 50 and K % g == 0
    assert bench.graph_calls(2000) == 50 and bench.graph_calls(97) == 1
