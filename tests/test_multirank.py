"""The N>1 host path of bench.py on CPU: two gloo ranks (replicas of the decode step,
weak scaling) -- the job's time is the slowest rank's, the rate counts every rank's
queries, and each replica gets its own synthetic problem."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    try:
        # rank r took 10 + r ms for the timed steps and 20 - r ms end to end
        got = bench.max_over_ranks([10.0 + rank, 20.0 - rank], world, "cpu")
        q.put((rank, got, bench.replica_seed(bench.SEED, rank)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_replica():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g for _, g, _ in res] == [[11.0, 20.0], [11.0, 20.0]]  # max over ranks, per timing
    seeds = [s for _, _, s in res]
    assert seeds[0] == 2 and len(set(seeds)) == world  # rank 0 keeps the workload seed


def test_job_rate_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    # 2 ranks x 32 queries x 400 steps in 200 ms
    assert bench.job_rate(2, 32, 400, 200.0) == pytest.approx(128000.0)
    assert bench.job_rate(1, 32, 400, 200.0) == pytest.approx(64000.0)
