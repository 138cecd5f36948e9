"""bench.py's multi-rank timing on CPU: two gloo ranks, each reporting its own
time; every rank must see the slowest rank's time, and the whole-job value is
the work of all ranks over that time.  (The GPU path runs one independent
replica of the training step per GPU; no collective is on the data path.)"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    val = bench.tflops(w, 1e12, 4, ms)
    q.put((r, w, lr, ms, val))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for (r, w, lr, ms, val) in out:
        assert w == 2 and r == lr
        assert ms == 15.0                      # the slower rank's 15 ms
        assert val == pytest.approx(2 * 1e12 * 4 / 0.015 / 1e12)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.tflops(1, 2e12, 10, 1000.0) == pytest.approx(20.0)
