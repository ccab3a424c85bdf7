"""Host logic of bench.py for N > 1 ranks, on the CPU with the gloo backend
(world_size 2): the barrier, the max-over-ranks of the step times, the head
partition (every head of the multi-rank problem owned by exactly one rank,
each rank's input block distinct) and the whole-job tokens/s (weak scaling:
the problem has world x H heads, H per rank)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    d = bench.Dist()
    try:
        d.barrier()
        ms = 1.0 + rank          # rank 1 is the slow one
        q.put((rank, d.max(ms), d.world))
        d.barrier()
    finally:
        d.close()


def test_two_rank_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(2))
    assert out == [(0, 2.0, 2), (1, 2.0, 2)]


def _partition_worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch
    import torch.distributed as dist
    import bench
    import kda_inputs as ki
    d = bench.Dist()
    try:
        w = ki.custom_workload(1, 64, 2, 32, 32, dtype="fp32", name="part")
        h0, h1 = bench.head_partition(w.H * d.world, d.world, d.rank)
        x = ki.make_inputs(w, seed=bench.head_block_seed(5, h0, w.H))
        heads = list(range(h0, h1))
        gathered = [None] * d.world
        dist.all_gather_object(gathered, (heads, x["q"].flatten()[:64].tolist()))
        q.put((rank, gathered))
        d.barrier()
    finally:
        d.close()


def test_two_rank_head_partition_covers_every_head_once():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_partition_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    outs = dict(q.get(timeout=10) for _ in range(2))
    for rank in (0, 1):
        parts = outs[rank]
        heads = sorted(h for hs, _ in parts for h in hs)
        assert heads == [0, 1, 2, 3]            # 2 ranks x 2 heads, each once
        assert parts[0][1] != parts[1][1]       # distinct input blocks


def test_head_partition_rejects_uneven_split():
    import bench
    assert bench.head_partition(32, 4, 3) == (24, 32)
    with pytest.raises(ValueError):
        bench.head_partition(30, 4, 0)


def test_whole_job_value_is_weak_scaling_sum():
    import bench
    # 2 replicas of 8192 tokens, slowest rank 1 ms -> 16.384 M tokens/s
    assert bench.whole_job_value(2, 8192, 1.0) == pytest.approx(16.384e6)
