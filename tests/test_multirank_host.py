"""The benchmark's multi-GPU path is N independent replicas (the GEMV does
not shard); its host logic — the slowest rank's time, the whole-job
throughput, rank 0 alone running the reference arm — checked with two gloo
ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.5, 5.25][rank]          # rank 1 is the slower replica
        got = bench.reduce_max(local_ms)
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out == {0: 5.25, 1: 5.25}


def test_single_process_reduce_is_identity():
    assert bench.reduce_max(2.5) == 2.5


def test_job_throughput_is_weak_scaling_over_the_slowest_rank():
    # 2 replicas, each 56.77 MB per step, 50 steps, slowest rank 2 ms
    assert bench.job_throughput(56.77e6, 50, 2, 2.0) == pytest.approx(56.77e6 * 100 / 2e-3 / 1e9)
    assert bench.job_throughput(1e9, 1, 1, 1000.0) == pytest.approx(1.0)


def test_reference_arm_on_other_ranks_exits_without_work():
    class A:
        steps, warmup = 1, 3
    assert bench.run_reference(A(), 1, 2) == 0
