"""Multi-rank host logic on CPU (gloo, world size 2).

Experts are independent units ("05 · Grouped GEMM 与 Expert 计算", introduction and section 2:
expert parallelism places each expert's tokens on one device). ``assign_experts`` places them on
ranks with balanced token sums; each rank computes its experts from its own slices of A and B
with no data-path exchange. The tests check the placement, that per-rank results reassembled
equal the single-rank result bit for bit, and the benchmark's timing reduction (the slowest
rank's time) and whole-job throughput.
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


# ------------------------------------------------------------------------------------------
# Expert placement
# ------------------------------------------------------------------------------------------

def test_assign_experts_places_each_expert_once_with_balanced_token_sums():
    import numpy as np

    from grouped_gemm_expert_gb300.partition import assign_experts, rank_token_sums
    rng = np.random.default_rng(5)
    for world in (1, 2, 3, 4, 8):
        for _ in range(20):
            counts = 256 * rng.integers(0, 40, size=int(rng.integers(1, 70)))
            owned = assign_experts(counts, world)
            assert len(owned) == world
            flat = sorted(e for o in owned for e in o)
            assert flat == list(range(len(counts)))
            assert all(o == sorted(o) for o in owned)
            sums = rank_token_sums(counts, owned)
            assert sum(sums) == int(counts.sum())
            assert max(sums) - min(sums) <= int(counts.max())      # list-scheduling bound
    assert assign_experts([5, 5, 5, 5], 2) == [[0, 2], [1, 3]]
    assert assign_experts([100, 1, 1, 1], 2) == [[0], [1, 2, 3]]
    with pytest.raises(ValueError):
        assign_experts([1, -1], 2)
    with pytest.raises(ValueError):
        assign_experts([1], 0)


def test_local_problem_lists_the_rank_experts_in_order():
    import numpy as np

    from grouped_gemm_expert_gb300.partition import local_problem
    counts = [256, 0, 512, 768]
    local, offsets, ranges = local_problem(counts, [1, 3])
    assert local.tolist() == [0, 768] and offsets.tolist() == [0, 768] and offsets.dtype == np.int32
    assert ranges == [(256, 256), (768, 1536)]


def _partition_worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np

    import oracle.kgw_oracle as O
    import workloads as W
    from grouped_gemm_expert_gb300.partition import assign_experts, local_problem
    counts = [256, 768, 0, 512, 1024, 256, 512]
    w = W.custom(len(counts), 128, 256, counts, seed=91)
    x = W.make_inputs(w, "cpu")
    a = x.a.view(torch.int16).numpy().view(np.uint16)      # [H, T] K-major
    b = x.b.view(torch.int16).numpy().view(np.uint16)      # [T, I] N-major
    mine = assign_experts(counts, world)[rank]
    local, offsets, ranges = local_problem(counts, mine)
    # this rank's tokens: its experts' columns of A and rows of B, back to back
    cols = np.concatenate([np.arange(lo, hi) for lo, hi in ranges]) if ranges else np.zeros(0, dtype=np.int64)
    a_loc, b_loc = np.ascontiguousarray(a[:, cols]), np.ascontiguousarray(b[cols, :])
    r_loc, _ = O.wgrad_from_storage(a_loc, b_loc, offsets, 128, 256)
    part = {e: r_loc[i] for i, e in enumerate(mine)}
    gathered = [None] * world
    dist.all_gather_object(gathered, part)
    if rank == 0:
        whole, _ = O.wgrad_from_storage(a, b, w.offsets, 128, 256)
        merged = {}
        for g in gathered:
            assert not set(g) & set(merged)
            merged.update(g)
        same = sorted(merged) == list(range(len(counts))) and all(
            np.array_equal(merged[e], whole[e]) for e in range(len(counts)))
        q.put(("ok" if same else "mismatch", [len(g) for g in gathered]))
    dist.barrier()
    dist.destroy_process_group()


def test_partitioned_experts_reassemble_to_the_single_rank_result():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_partition_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    verdict, sizes = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert verdict == "ok"
    assert sum(sizes) == 7 and min(sizes) >= 1
