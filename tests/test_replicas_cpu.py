"""The benchmark's multi-rank logic on CPU: two gloo ranks (replicas, no
data-path collective) agree on the slowest rank's time, and the job's rate
counts every rank's units over that time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.0, 3.5][rank]                         # rank 1 is the slow one
    got = bench.reduce_max_over_ranks(dist, ms, "cpu")
    rate = bench.whole_job_rate(1e9, got, world)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, got, rate))


def test_two_gloo_ranks_max_time_and_job_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate in res:
        assert got == 3.5                               # max over ranks, on every rank
        assert rate == pytest.approx(2 * 1e9 / 3.5e-3)  # both ranks' units / slowest time


def test_single_process_passthrough():
    import bench
    assert bench.reduce_max_over_ranks(None, 1.25, "cpu") == 1.25
    assert bench.whole_job_rate(10.0, 2.0, 1) == pytest.approx(5000.0)
