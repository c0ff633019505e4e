"""The benchmark's multi-rank arithmetic (replicas: max over ranks of the step
time, throughput summed over ranks), run as two gloo ranks on the CPU."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.reduce_step_time(1.0 + rank, world)   # rank 1 is slower
    q.put((rank, ms, bench.job_throughput(10 ** 9, ms, world)))
    dist.destroy_process_group()


def test_two_rank_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    assert [r[1] for r in res] == [2.0, 2.0]
    assert res[0][2] == pytest.approx(2 * 10 ** 9 / 2e-3 / 1e9)


def test_single_rank_is_identity():
    assert bench.reduce_step_time(3.5, 1) == 3.5
    assert bench.job_throughput(10 ** 9, 1.0, 1) == pytest.approx(1000.0)
