"""The N > 1 path of bench.py, on the CPU: two ranks over gloo (world size 2).

Each GPU runs an independent replica (the path has no exchange between GPUs); the job's
time is the slowest rank's, taken with an all-reduce max, and its rate is all ranks' FLOPs
over that time.  The reference arm runs on rank 0 only; other ranks exit without output.
"""

import argparse
import contextlib
import io
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slow = bench.dist_max(10.0 * (rank + 1), world)      # rank 1 is the slow one
    bench.dist_barrier(world)
    rate = bench.job_rate(world, 3.0e12, 4, slow)
    buf = io.StringIO()
    args = argparse.Namespace(steps=1, warmup=0)
    with contextlib.redirect_stdout(buf):
        if rank != 0:
            bench.run_reference(args, bench.workload("32k", None), rank, world)
    q.put((rank, slow, rate, buf.getvalue()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slow, rate, out in res:
        assert slow == 20.0
        # 2 ranks x 4 steps x 3e12 FLOP over 20 ms
        assert rate == pytest.approx(2 * 4 * 3.0e12 / 0.020 / 1e12)
        if rank != 0:
            assert out == ""
