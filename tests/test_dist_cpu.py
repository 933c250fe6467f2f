"""bench.py's multi-rank plumbing on CPU: two gloo ranks, barrier and max-over-ranks timing.

The hot path does not exchange data between GPUs (independent trees run as
replicas); the only cross-rank steps are the barrier around the timed region
and the maximum of the per-rank times, which these ranks exercise.
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
    # CPU ranks even on a machine with GPUs (gloo; a second rank would find no second GPU)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    import bench
    r, w, _ = bench.dist_setup(world)
    bench.barrier(w)
    got = bench.max_over_ranks(10.0 + 5.0 * r, w)
    q.put((r, w, got))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_max_and_barrier():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=120) for _ in procs)
        for p in procs:
            p.join(timeout=60)
            assert p.exitcode == 0
    finally:
        for p in procs:  # a rank that failed must not leave its peer waiting in the rendezvous
            if p.is_alive():
                p.terminate()
                p.join(timeout=10)
    assert res == [(0, 2, 15.0), (1, 2, 15.0)]


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
