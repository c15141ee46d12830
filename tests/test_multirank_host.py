"""The N > 1 bench logic on CPU: two gloo ranks, no GPU.

The workload shards by batch/channel with no data-path collective, so the
only cross-rank step is the timing reduction (max over ranks) and the
whole-job aggregation of bytes.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = 10.0 + 5.0 * rank
    got = bench.max_over_ranks(mine)
    dist.barrier()
    q.put((rank, got, bench.whole_job_gbps(1e9, 4, world, got)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, gbps in res:
        assert got == pytest.approx(15.0)
        assert gbps == pytest.approx(world * 4 * 1e9 / 0.015 / 1e9)


def test_single_rank_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_gbps(2e9, 10, 1, 1000.0) == pytest.approx(20.0)
