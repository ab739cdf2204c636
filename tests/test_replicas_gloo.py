"""The N > 1 host logic of the benchmark on CPU: world-size-2 gloo ranks
reduce their step times (max) and work (sum) the way bench.py's replicas do."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t, u = bench.reduce_time_units(10.0 + rank * 5.0, 100.0 * (rank + 1), torch.device("cpu"), world)
    results[rank] = (t, u)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_reduce_like_the_benchmark():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert results[0] == results[1] == (15.0, 300.0)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_time_units(3.0, 7.0, torch.device("cpu"), 1) == (3.0, 7.0)
