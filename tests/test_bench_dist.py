"""The benchmark's multi-rank plumbing on CPU: two gloo ranks (the layout
torchrun gives one process per GPU).  Each rank reports its own timing; the
step time is the maximum over ranks, and only rank 0 prints."""
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
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import bench

    r, w = bench.dist_init("gloo")
    bench.barrier(None)
    got = bench.max_over_ranks(10.0 + 5.0 * rank)
    q.put((r, w, got))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert res == [(0, 2, 15.0), (1, 2, 15.0)]


def test_single_process_has_no_group():
    sys.path.insert(0, ROOT)
    import bench

    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        if k in os.environ:
            pytest.skip("running under a launcher")
    assert bench.dist_init("gloo") == (0, 1)
    assert bench.max_over_ranks(3.5) == 3.5
