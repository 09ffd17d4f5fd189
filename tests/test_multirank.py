"""The N>1 path of bench.py on the CPU: two gloo ranks run independent
replicas and agree on the max step time over ranks (the only cross-rank
exchange; nothing on the data path)."""
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


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.dist_barrier(world)
        local_ms = 1.0 + rank * 0.5          # each replica measures its own time
        results[rank] = bench.dist_max(local_ms, world)
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_take_the_max_time():
    world = 2
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(results) == {0: 1.5, 1: 1.5}
