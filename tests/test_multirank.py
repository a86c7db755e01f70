"""Multi-process plumbing of bench.py on CPU (gloo, world size 2).

Rows are independent, so several GPUs run independent replicas with no
collective on the data path; the benchmark only needs a barrier around the
timed region and the maximum of the per-rank times.  This is exercised here
with two CPU processes.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    ws, r, local = bench.dist_setup()
    assert (ws, r, local) == (world, rank, rank)
    mine = 1.5 * (rank + 1)
    bench.barrier(ws)
    got = bench.max_over_ranks(mine, ws)
    # the reference arm: only rank 0 does work, the others return at once
    class A:
        workload = "tiny"; steps = 1; warmup = 0
    if rank != 0:
        bench.run_reference(A, ws, rank)
    bench.barrier(ws)
    q.put((rank, got))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_barrier_and_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("rank did not finish")
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r for r, _ in res] == [0, 1]
    assert all(abs(v - 3.0) < 1e-12 for _, v in res)
