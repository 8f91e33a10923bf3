"""The N > 1 host logic of bench.py (replicas, weak scaling), as two gloo ranks on CPU: the barrier,
the max over ranks (the job's time is its slowest rank's), the whole-job throughput, and the
reference arm running on rank 0 only."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    bench._PG = dist.group.WORLD
    bench._PG_DEVICE = "cpu"
    bench.barrier()
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank)  # rank 1 is the slow one
    value = bench.job_throughput_gbs(65_667_584, 1000, slowest, world)
    out = io.StringIO()
    with contextlib.redirect_stdout(out):

        class A:
            steps, warmup = 1, 0

        rc = bench.run_reference(A) if rank == 1 else 0  # rank 1 must exit without work
    q.put((rank, slowest, value, rc, out.getvalue()))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value, rc, out in res:
        assert slowest == 15.0
        assert value == pytest.approx(2 * 65_667_584 * 1000 / 15e-3 / 1e9)
        assert rc == 0 and out == ""


def test_single_rank_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput_gbs(1_000_000_000, 10, 1000.0, 1) == pytest.approx(10.0)
