"""The multi-GPU form of the bench is N independent replicas (every (sequence, head) is
independent, so nothing is exchanged); ranks meet only to take the slowest rank's time.
This checks that reduction and the whole-job rate with two gloo ranks on the CPU."""
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


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r took (r + 1) ms for prefill and 10 (r + 1) us for decode
        got = bench.max_over_ranks([1e-3 * (rank + 1), 10e-6 * (rank + 1)], torch.device("cpu"))
        dist.barrier()
        q.put((rank, got, bench.job_throughput(world, 4096, got[0])))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, got, rate in res:
        assert got == pytest.approx([2e-3, 20e-6])
        assert rate == pytest.approx(2 * 4096 / 2e-3)
