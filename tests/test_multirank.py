"""Multi-process host logic of the benchmark (CPU, gloo, world size 2).

Every rank runs its own replica of the workload (weak scaling, no collective in
the data path); the job's time is the slowest rank's and the job's throughput
counts the work of all ranks.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [10.0, 14.0][rank]
    ms = bench.max_over_ranks(local_ms)
    q.put((rank, ms, bench.job_tflops(2e12, ms, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_time_and_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tf in res:
        assert ms == 14.0                     # the slowest rank sets the time
        assert abs(tf - 2 * 2e12 / 14e-3 / 1e12) < 1e-9  # both ranks' work counts


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tflops(1e12, 1000.0, 1) == pytest.approx(1.0)
