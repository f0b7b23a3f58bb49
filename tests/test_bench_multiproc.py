"""The benchmark's multi-rank host logic on CPU with the gloo backend
(world size 2): batch ownership per rank, max-over-ranks timing, and the
whole-job throughput aggregation."""

import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        elapsed = 1.0 + rank  # rank 1 is the slow one
        bench.barrier(world)
        mx = bench.max_over_ranks(elapsed, world)
        q.put((rank, mx, bench.rank_batch_range(rank, 22)))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_timing_and_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [m for _, m, _ in res] == [2.0, 2.0]          # max over ranks on every rank
    assert res[0][2] == (0, 22) and res[1][2] == (22, 44)  # disjoint batches, weak scaling
    sys.path.insert(0, ROOT)
    import bench

    # whole-job tokens/s: both ranks' tokens over the slowest rank's time
    assert bench.whole_job_throughput(22 * 512, 2, 10, 2.0) == pytest.approx(22 * 512 * 2 * 10 / 2.0)
    assert bench.counted_flops(22, 8, 64, 512, 512) == 26_592_411_648
