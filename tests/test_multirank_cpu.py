"""The N > 1 host path of bench.py on CPU: two gloo ranks, each a replica
with its own step time; the job reports the slowest rank and the summed
throughput.  No GPU, no data-path collective (the path shards into replicas)."""

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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 2.0 + rank  # rank 1 is the slower replica
    worst = bench.max_over_ranks(ms, world)
    value = bench.aggregate_tflops(1e12, worst, world)
    dist.barrier()
    out[rank] = (worst, value)
    dist.destroy_process_group()


def test_two_gloo_ranks_max_and_aggregate():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        worst, value = out[r]
        assert worst == 3.0
        assert value == pytest.approx(2 * 1e12 / 3e-3 / 1e12)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.aggregate_tflops(2e12, 1.0, 1) == pytest.approx(2000.0)
