"""The multi-process path of bench.py on CPU: two gloo ranks, each timing its own replica.

bench.py under torchrun runs one independent replica per rank (the sublayer needs no exchange between
GPUs); the job's value is every rank's tokens over the slowest rank's time.  This checks the barrier,
the max-over-ranks reduction and the aggregation with world_size 2.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench

    ws, r, local = bench.dist_setup()
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    seconds = 0.5 + rank  # rank 1 is the slow one
    slowest = bench.max_over_ranks(seconds, ws)
    out[rank] = (slowest, bench.aggregate(16384, ws, slowest))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    port = _free_port()
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(2):
            slowest, value = out[r]
            assert slowest == pytest.approx(1.5)
            assert value == pytest.approx(2 * 16384 / 1.5)


def test_single_rank_defaults():
    import bench

    assert bench.max_over_ranks(2.0, 1) == 2.0
    assert bench.aggregate(100, 1, 0.5) == 200.0
