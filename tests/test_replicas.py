"""Host logic of bench.py with N > 1 processes (replicas only: no data-path
collective), as world_size-2 gloo ranks on the CPU: rendezvous, the barrier
around the timed region, the max-over-ranks time, and the reference arm that
only rank 0 runs."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    # per-rank elapsed times; every rank must see the slowest one
    m = bench.max_over_ranks(0.25 + 0.5 * r, w, torch.device("cpu"))
    bench.barrier(w)
    # the reference arm: rank != 0 returns at once, without touching the oracle
    if r != 0:
        class A:
            pass
        bench.run_reference(A(), w, r)
    q.put((r, w, m))
    torch.distributed.destroy_process_group()


def test_two_replicas_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.terminate()
    assert codes == [0, 0], codes
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == world for g in got)
    assert all(g[2] == pytest.approx(0.75) for g in got)   # max over ranks


def test_single_process_helpers_are_noops():
    sys.path.insert(0, ROOT)
    import bench

    bench.barrier(1)
    assert bench.max_over_ranks(1.5, 1, torch.device("cpu")) == 1.5
