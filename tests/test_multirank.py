"""The benchmark's multi-rank logic on CPU with the gloo backend, world size 2:
each rank times its own units, the job time is the slowest rank's, and the
job throughput counts every rank's units. No collective touches the data path."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys

    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    got = bench.max_over_ranks(ms, "cpu")
    dist.barrier()
    out.put((rank, got, bench.job_value(1000.0, world, 4, got)))
    dist.destroy_process_group()


def test_two_ranks_gloo_max_time_and_job_throughput():
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
    for rank, got, value in res:
        assert got == pytest.approx(15.0)
        assert value == pytest.approx(1000.0 * 2 * 4 / 0.015)
