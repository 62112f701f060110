"""The benchmark's multi-rank bookkeeping on CPU: world size 2 over gloo. Each rank reports its
own units and time; the whole-job value is all ranks' units over the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist = bench.dist_init("gloo")
    units = 1000.0 * (rank + 1)
    seconds = 2.0 if rank == 0 else 4.0
    value, smax = bench.aggregate(dist, units, seconds)
    bench.barrier(dist)
    out[rank] = (value, smax)
    dist.destroy_process_group()


def test_aggregate_world2_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        value, smax = out[r]
        assert smax == pytest.approx(4.0)
        assert value == pytest.approx(3000.0 / 4.0)


def test_aggregate_single_process():
    value, smax = bench.aggregate(None, 500.0, 2.0)
    assert value == 250.0 and smax == 2.0


def test_alg_bytes_formula():
    # 68 B per key, 4 B per page-table entry, 72 B per query head, 8 B per output slot
    assert bench.decode_alg_bytes([131072] * 16, 64, 2048) == 16 * (68 * 131072 + 4 * 2048 + 64 * 72 + 2048 * 8)
    assert bench.decode_alg_bytes([1], 16, 64) == 68 + 4 + 16 * 72 + 64 * 8
