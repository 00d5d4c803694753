"""The benchmark's multi-GPU path (weak scaling: every rank runs the same
per-GPU workload, no collective on the data path, the slowest rank bounds the
job) exercised with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) seconds for decode and (2 - r) for extend
        dec, ext, loop = bench.max_over_ranks([rank + 1.0, 2.0 - rank, 10.0 + rank], dist)
        value = bench.weak_scaling_throughput(world, 100, 1e9, dec)
        dist.barrier()
        q.put((rank, dec, ext, loop, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_two_gloo_ranks():
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
    for rank, dec, ext, loop, value in res:
        assert (dec, ext, loop) == (2.0, 2.0, 11.0)        # every rank sees the slowest rank
        assert value == pytest.approx(2 * 100 * 1e9 / 2.0)  # both ranks' units over the max time


def test_single_process_is_identity():
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.weak_scaling_throughput(1, 10, 5.0, 2.0) == 25.0
