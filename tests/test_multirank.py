"""The benchmark's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

Each rank runs its own batch (weak scaling); the only collective is the
max-over-ranks of the timed region, and the whole-job value counts every
rank's tokens against that slowest time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, dist)   # rank 1 is the slow one
    value = bench.weak_scaling_value(64, world, 100, slowest)
    out.put((rank, slowest, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in res:
        assert slowest == pytest.approx(15.0)
        assert value == pytest.approx(64 * 2 * 100 / 15e-3)


def test_single_rank_needs_no_collective():
    import bench

    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.weak_scaling_value(64, 1, 10, 2.0) == pytest.approx(64 * 10 / 2e-3)
