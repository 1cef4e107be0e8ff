"""The multi-GPU path is replicas only: every rank runs the same layer step on its own GPU
and the bench reports the slowest rank's time and the whole job's throughput.  These tests
run that host logic as two gloo ranks on the CPU (no GPU)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        slowest = bench.max_over_ranks(times[rank], dist)
        value = bench.replica_throughput(world, 8, 100, slowest)
        t = torch.tensor([slowest, value], dtype=torch.float64)
        gathered = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(gathered, t)
        if rank == 0:
            out.put([g.tolist() for g in gathered])
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    times = [8.0, 10.0]  # ms for 100 steps on rank 0 and rank 1
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = q.get()
    # every rank agrees on the slowest time and on the whole job's throughput
    assert all(r[0] == pytest.approx(10.0) for r in res)
    expect = 2 * 8 * 100 / (10.0 / 1000.0)
    assert all(r[1] == pytest.approx(expect) for r in res)


def test_one_process_needs_no_collective():
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.replica_throughput(1, 8, 10, 2.0) == pytest.approx(8 * 10 / 0.002)
