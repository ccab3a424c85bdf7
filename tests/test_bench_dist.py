"""Host logic of bench.py for N > 1 ranks, on the CPU with the gloo backend
(world_size 2): the barrier, the max-over-ranks of the step times and the
whole-job tokens/s (every rank runs its own replica: weak scaling)."""
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


def test_whole_job_value_is_weak_scaling_sum():
    import bench
    # 2 replicas of 8192 tokens, slowest rank 1 ms -> 16.384 M tokens/s
    assert bench.whole_job_value(2, 8192, 1.0) == pytest.approx(16.384e6)
