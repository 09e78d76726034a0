"""bench.py's multi-GPU host logic on CPU: two ranks over gloo. Each rank
runs its own replica (weak scaling); the ranks only meet in the barrier
around the timed region and in the max of their step times, and only rank 0
runs the CPU reference arm."""
import io
import multiprocessing
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    ranks = bench.Ranks(backend="gloo")
    ranks.barrier()
    slowest = ranks.max(10.0 + rank)           # per-rank step times 10 ms and 11 ms
    # the reference arm: rank 0 alone works; the others return at once
    out = io.StringIO()
    if rank != 0:
        with redirect_stdout(out):
            bench.run_reference(type("A", (), {"steps": 1, "warmup": 0, "cpu_budget": 0.1})())
    ranks.barrier()
    queue.put((rank, ranks.world, slowest, out.getvalue()))
    ranks.close()


def test_two_gloo_ranks_take_the_slowest_step_time():
    ctx = multiprocessing.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = [queue.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    assert [r[1] for r in results] == [2, 2]
    assert [r[2] for r in results] == [11.0, 11.0]
    assert results[1][3] == ""                 # rank 1 printed no reference line


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    ranks = bench.Ranks()
    assert ranks.world == 1 and ranks.max(3.5) == 3.5
