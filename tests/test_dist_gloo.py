"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

Experts are independent, so N ranks run N independent batches with no data-path exchange; the
only collective is the timing reduction (the slowest rank's time) and the whole-job
throughput counts every rank's work.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    t = bench.max_over_ranks(1.0 + rank * 0.5, world, "cpu")
    thr = bench.job_throughput(2e12, t, world)
    q.put((rank, t, thr))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_work():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, thr in res:
        assert t == pytest.approx(1.5)
        assert thr == pytest.approx(2 * 2e12 / 1.5e-3 / 1e12)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_throughput(1e12, 1.0, 1) == pytest.approx(1000.0)
