"""Host logic of the multi-process bench on CPU: two gloo ranks.

Decode shards by batch element with no exchange between ranks (each rank
decodes its own batch), so the only cross-rank step is the timing reduction:
the job time is the slowest rank's, and throughput counts every rank's units.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 * (rank + 1)           # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, "cpu")
        value = bench.job_throughput(1000.0, world, ms)
        q.put((rank, ms, value, bench.rank_seed("dense_membound", rank)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value, seed in res:
        assert ms == pytest.approx(20.0)                 # max over ranks, seen by every rank
        assert value == pytest.approx(2 * 1000.0 / 20e-3)  # both ranks' units over the slowest time
    assert res[0][3] != res[1][3]                        # ranks decode different batches
    assert res[0][3] == bench.W.SEEDS["dense_membound"]  # rank 0 is the single-GPU workload


def test_single_process_reduction_is_identity():
    assert not (dist.is_available() and dist.is_initialized())
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.job_throughput(10.0, 1, 2.0) == pytest.approx(5000.0)
