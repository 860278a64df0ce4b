"""bench.py's multi-rank plumbing on the CPU: two gloo ranks, the same calls
the timed region makes (process-group set-up from the torchrun environment,
barrier, max over ranks of the elapsed time), and the reference arm's rule
that only rank 0 produces a line."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    try:
        w, r, local = bench.dist_setup()
        assert (w, r, local) == (world, rank, rank)
        bench.barrier(w)
        m = bench.allreduce_max(1.5 + rank * 2.25, w)
        bench.barrier(w)

        class A:
            config, steps, warmup, gpus = "tiny", 1, 3, world
        ref = bench.run_reference(A, w, r) if r != 0 else "skipped"
        q.put((rank, m, ref))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    got = sorted(q.get(timeout=5) for _ in range(world))
    # every rank sees the max over ranks
    assert [g[1] for g in got] == [1.5 + 2.25, 1.5 + 2.25]
    # the reference arm does no work on ranks other than 0
    assert got[1][2] is None


def test_single_rank_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.allreduce_max(3.25, 1) == 3.25
    bench.barrier(1)
