"""Host logic of the multi-rank bench run (weak-scaling replicas, no data-path
collective), on two gloo ranks on the CPU: the job's time is the slowest rank's, and the
job's throughput counts every rank's steps."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q) -> None:
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured (10 + r) ms for the timed steps and (30 - r) ms for e2e
        got = bench.max_over_ranks([10.0 + rank, 30.0 - rank], dist, device="cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [11.0, 30.0]


def test_single_rank_and_job_throughput():
    assert bench.max_over_ranks([3.5, 7.0], None) == [3.5, 7.0]
    # 2 ranks x 4 steps x 1e12 flops in 2 ms -> 4000 TFLOPS
    assert bench.job_tflops(2, 10 ** 12, 4, 2.0) == pytest.approx(4000.0)
