"""Host logic of bench.py's multi-GPU (replica) mode on CPU: two gloo ranks,
max-over-ranks timing and the whole-job value."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (rank, world, rank)
    ms = bench.reduce_max(1.5 + rank, device="cpu")
    q.put((rank, ms, bench.job_value(ms, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(2))
    assert [g[1] for g in got] == [2.5, 2.5]
    assert [g[2] for g in got] == [1250.0, 1250.0]


def test_single_process_value():
    import bench

    assert bench.reduce_max(3.0) == 3.0
    assert bench.job_value(2.0, 1) == 2000.0
