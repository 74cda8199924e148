"""The multi-rank logic of bench.py on CPU with the gloo backend (world size 2):
timing is reduced with MAX over ranks and the reported value aggregates every
rank's replica (weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_info()
        assert (r, w, lr) == (rank, world, rank)
        elapsed = 10.0 + 5.0 * rank           # rank 1 is the slow one
        bench.barrier(world)
        m = bench.max_over_ranks(elapsed, world)
        q.put((rank, m, bench.aggregate_value(world, 16, 4, m)))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, value in out:
        assert m == 15.0                                   # max over ranks
        assert value == pytest.approx(2 * 16 * 4 / 0.015)  # both replicas, slowest clock


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate_value(1, 16, 10, 1000.0) == 160.0
