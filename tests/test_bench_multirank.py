"""The bench's multi-rank host logic on CPU: two gloo ranks, each timing its
own replica of the workload (weak scaling), agree on the slowest rank's time
and report the whole-job rate over both ranks."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.cpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured (2 + r) ms for the step loop and (10 - r) ms end to end
        got = bench.max_over_ranks([2.0 + rank, 10.0 - rank], world)
        rate = bench.whole_job_rate(34, 4, world, got[0])
        queue.put((rank, got, rate))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_units():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, got, rate in res:
        assert got == [3.0, 10.0], (rank, got)
        # 34 layer-steps x 4 steps on each of 2 ranks in 3 ms
        assert rate == pytest.approx(34 * 4 * 2 / 3e-3)


def test_one_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.whole_job_rate(64, 100, 1, 6.0) == pytest.approx(64 * 100 / 6e-3)

