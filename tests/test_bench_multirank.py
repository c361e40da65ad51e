"""Host logic of bench.py's multi-GPU mode (independent replicas, weak
scaling) on CPU: two gloo ranks, the step time is the maximum over ranks and
the job's throughput counts every rank's work. No collective touches the
layer's data path."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    m = bench.reduce_max(ms)
    dist.barrier()
    q.put((rank, m, bench.job_metrics(world, m, 1e12, 4096)))
    dist.destroy_process_group()


def test_two_rank_replicas_aggregate_by_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for rank, m, jm in res:
        assert m == 15.0
        assert jm["tflops"] == pytest.approx(2 * 1e12 / 15e-3 / 1e12)
        assert jm["tokens_per_s"] == pytest.approx(2 * 4096 / 15e-3)


def test_single_process_needs_no_process_group():
    assert bench.reduce_max(3.5) == 3.5
    jm = bench.job_metrics(1, 2.0, 1e12, 100)
    assert jm["tflops"] == pytest.approx(500.0) and jm["tokens_per_s"] == pytest.approx(5e4)
