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


def test_reference_arm_json_line_on_cpu():
    """`bench.py --impl reference` times the oracle on the host cores and prints
    one JSON line in the bench contract (no GPU needed)."""
    import json
    import subprocess
    import sys
    res = subprocess.run([sys.executable, os.path.join(REPO, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "1", "--warmup", "3", "--reference-budget", "2"],
                         capture_output=True, text=True, timeout=600, cwd=REPO)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GB/s"
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config"):
        assert key in line, key
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
