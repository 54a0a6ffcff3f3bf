"""bench.py's multi-process plumbing on CPU: two gloo ranks (no GPU).

Each rank runs its own replica of the workload (weak scaling): the seeds must
differ per rank, `max` must return the slowest rank's time and `sum` the
whole job's bytes on every rank.
"""
import os
import socket

import torch.multiprocessing as mp

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import sys
    sys.path.insert(0, REPO)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    ctx = bench.DistCtx()
    try:
        wl = bench.workload_for("tiny", ctx.rank)
        ctx.barrier()
        results[rank] = (ctx.max(1.0 + rank), ctx.sum(10.0 * (rank + 1)), wl.seed)
    finally:
        ctx.close()


def test_two_gloo_ranks_reduce_and_use_distinct_seeds():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank, args=(world, port, results), nprocs=world, join=True,
                           start_method="spawn")
        got = dict(results)
    assert got[0][0] == got[1][0] == 2.0
    assert got[0][1] == got[1][1] == 30.0
    assert got[0][2] != got[1][2]
