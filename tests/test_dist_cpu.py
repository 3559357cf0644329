"""The multi-rank measurement path of bench.py on CPU (world size 2, gloo):
weak scaling sums the bytes of all ranks and divides by the slowest rank's
time; the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r moved (r + 1) GB in (r + 1) seconds
        value, t = bench.aggregate((rank + 1) * 1e9, float(rank + 1), world)
        mx = bench.max_over_ranks(float(10 * rank), world)
        sm = bench.sum_over_ranks(float(rank + 1), world)
        bench.barrier(world)
        q.put((rank, value, t, mx, sm))
    finally:
        dist.destroy_process_group()


def test_weak_scaling_aggregate_two_ranks():
    import multiprocessing as mp
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
    for rank, value, t, mx, sm in res:
        assert t == 2.0                      # slowest rank
        assert value == pytest.approx(1.5)   # (1 + 2) GB over the slowest 2 s
        assert mx == 10.0 and sm == 3.0


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(5e9, 2.0, 1) == (2.5, 2.0)
