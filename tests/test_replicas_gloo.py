"""bench.py's multi-GPU path is N independent replicas (the verify step of
one request does not shard without the pages' tensor parallelism): every
rank runs its own step, the timed region is bracketed by barriers, the job
time is the slowest rank's, and the throughput sums all ranks' tokens.  This
runs that host logic with two gloo ranks on the CPU (no GPU)."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "MSK_BENCH_BACKEND": "gloo"})
    import bench
    rk = bench.Ranks()
    try:
        rk.barrier()
        my_time = 1.0 + 0.5 * rank  # rank 1 is the slow one
        slowest = rk.max(my_time)
        rk.barrier()
        q.put((rank, rk.world, slowest, bench.aggregate(slowest, 16 * 20, rk.world)))
    finally:
        rk.close()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_and_sum_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=5) for _ in range(2))
    for rank, world, slowest, value in out:
        assert world == 2
        assert slowest == 1.5  # the max over ranks, seen identically by every rank
        assert value == pytest.approx(16 * 20 * 2 / 1.5)  # all ranks' tokens over the slowest time


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    rk = bench.Ranks()
    assert rk.world == 1 and rk.dist is None
    assert rk.max(3.25) == 3.25
    rk.barrier()
    rk.close()
