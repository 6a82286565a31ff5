"""The benchmark's multi-rank path on CPU ranks (gloo, world size 2): every rank
times its own copy of the workload, the reported time is the slowest rank's,
and the value counts the elements of all ranks."""

import os
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier(world)
        ms = 10.0 + 5.0 * rank                     # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, world, "cpu")
        value = bench.weak_scaling_value(1e9, world, slowest)
        bench.rank_barrier(world)
        out.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, 29500 + os.getpid() % 1000
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]
    # 1e9 elements per rank, two ranks, 15 ms: 133.3 Gelem/s whole-job
    assert res[0][2] == pytest.approx(2e9 / 0.015 / 1e9)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    bench.rank_barrier(1)
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.weak_scaling_value(1e9, 1, 10.0) == pytest.approx(100.0)
