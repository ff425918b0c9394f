"""Multi-rank host logic of bench.py on CPU: two gloo ranks, the reported
step time is the max over ranks and the throughput counts every rank's
(independent) problem."""

import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (world, rank, rank)
    my_ms = [3.0, 5.5][rank]
    got = bench.reduce_max(my_ms, world)
    bench.barrier(world)
    results[rank] = got
    dist.destroy_process_group()


def test_two_rank_max_reduction():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, results))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(results) == {0: 5.5, 1: 5.5}


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max(1.25, 1) == 1.25
    a = bench.parse_args([])
    assert a.gpus == 1 and a.impl == "ours"
    assert a.workload == "cfg3_packed_s8192_d128"
