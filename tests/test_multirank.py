"""The benchmark's N>1 path on CPU: two gloo ranks, each timing its own
replica; the job time is the max over ranks and the work the sum."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist = bench.init_dist(world, "gloo")
    t = bench.max_over_ranks(10.0 + rank, world)
    w = bench.sum_over_ranks(100.0 * (rank + 1), world)
    ws, r, _ = bench.dist_env()
    bench.barrier(world)
    q.put((r, ws, t, w))
    dist.destroy_process_group()


def test_two_rank_aggregation():
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
    assert res == [(0, 2, 11.0, 300.0), (1, 2, 11.0, 300.0)]
