"""The benchmark's multi-rank path (one replica per GPU, no data-path
collective): the step time is the slowest rank's and the job throughput sums
all replicas.  Run as two gloo ranks on the CPU."""
import os
import socket

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
        ms = [1.25, 2.5][rank]  # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, dist, "cpu")
        value = bench.job_throughput(100.0, slowest * 1e-3, world)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 2.5
        assert abs(value - 2 * 100.0 / 2.5e-3) < 1e-6


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.0) == 3.0
    assert bench.job_throughput(10.0, 2.0, 1) == 5.0
