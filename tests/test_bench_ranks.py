"""bench.py's multi-rank timing on CPU: two gloo ranks, the slowest rank's time
and the whole-job throughput (replicas, no data-path collective)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    tmax, value = bench.aggregate(1.0 + rank, 1024 * 10, world)
    q.put((rank, tmax, value))
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    import torch.multiprocessing as mp
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
    for rank, tmax, value in res:
        assert tmax == 2.0                       # the slower rank
        assert value == 2 * 1024 * 10 / 2.0      # units of both ranks / slowest time


def test_aggregate_single_rank():
    import bench
    assert bench.aggregate(0.5, 1024, 1) == (0.5, 2048.0)
