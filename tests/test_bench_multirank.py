"""bench.py's N>1 path on the CPU: two gloo ranks, barrier and max over ranks.

With several GPUs the bench runs one independent replica per rank (the path
shards by stream with no exchange); the only cross-rank steps are the barrier
around the timed region and the max of the ranks' times, tested here."""

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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    t = bench.max_over_ranks(dist, torch, 1.5 + rank)      # this rank's "time"
    out[rank] = t
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 2.5


def test_single_rank_max_is_identity():
    import bench
    assert bench.max_over_ranks(None, torch, 3.25) == 3.25
