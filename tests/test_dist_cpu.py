"""The benchmark's multi-rank path, on CPU with the gloo backend (world size 2).

Every rank runs an independent replica (the decode shards by sequence and KV
head with no exchange step); the ranks only meet at barriers and at the
max-over-ranks of the timed region, and the reported value is the units all
ranks processed divided by that maximum.
"""
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

    ctx = bench.DistCtx()
    ctx.init("gloo")
    ctx.barrier()
    # rank r "took" 10 + 5r ms for its replica of 3 calls of B = 4 tokens
    t_max = ctx.max(10.0 + 5.0 * rank)
    units = ctx.sum(3 * 4)
    value = units / (t_max / 1e3)
    ctx.barrier()
    ctx.close()
    q.put((rank, t_max, units, value))


@pytest.mark.timeout(120)
def test_replicas_max_over_ranks_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=100) for _ in range(world)]
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, t_max, units, value in res:
        assert t_max == 15.0          # the slowest rank sets the time
        assert units == 24            # both replicas' work counts
        assert abs(value - 24 / 0.015) < 1e-6
