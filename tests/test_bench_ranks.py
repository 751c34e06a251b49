"""The multi-rank timing rule of bench.py on CPU with two gloo ranks: the job
time is the slowest rank's (all-reduce MAX) and the whole-job µs per call
divides it by every rank's calls.  (The GEMV path itself runs as independent
replicas, one per GPU, with no collective on the data path.)"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(10.0 + 3.0 * rank)  # rank 1 is the slower one
    dist.barrier()
    out.put((rank, ms, bench.job_us_per_call(ms, 4, world)))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_and_count_every_call():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, us in results:
        assert ms == 13.0, (rank, ms)
        assert us == 13.0 * 1e3 / (4 * 2), (rank, us)


def test_single_process_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.job_us_per_call(7.5, 4, 1) == 7.5e3 / 4
