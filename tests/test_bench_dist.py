"""bench.py's multi-process plumbing on CPU: world size 2 over gloo.

Each rank times its own replica; the job's time is the max over ranks and
the work is the sum, with no data-path collective."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.dist_barrier(w)
    mx = bench.dist_max(w, 1.5 + rank)          # rank-dependent "time"
    sm = bench.dist_sum(w, 10.0 * (rank + 1))   # rank-dependent "work"
    out.put((rank, mx, sm))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_replica_timing_max_and_sum_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.5, 30.0), (1, 2.5, 30.0)]


def test_single_process_helpers_are_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(1, 3.0) == 3.0 and bench.dist_sum(1, 4.0) == 4.0
