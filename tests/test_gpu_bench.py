"""bench.py's own arm on a GPU, shortened: the JSON line carries the keys of
the bench contract, the roofline is consistent with its own numbers, and the
line ends with the compact per-workload targets (needs a GPU)."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_bench_line_keeps_the_contract():
    res = subprocess.run(
        [sys.executable, os.path.join(REPO, "bench.py"), "--steps", "5", "--warmup", "3",
         "--no-trace", "--no-cpu-baseline", "--e2e-steps", "3", "--repeats", "2",
         "--gate-reps", "10"],
        capture_output=True, text=True, timeout=900, cwd=REPO)
    assert res.returncode == 0, res.stderr[-3000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "clocks",
                "e2e", "gpu_launches", "roofline"):
        assert key in line, key
    assert line["steps"] == 5 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["config"]["workload"].startswith("longctx_splitk")
    assert line["gpu_launches"] == 3 * 5          # append_tokens, decode, merge per step
    r = line["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert abs(r["achieved"] - r["algorithmic_bytes_per_launch"] / r["decode_ms"] / 1e6) < 1e-6 * r["achieved"]
    assert r["decode_ms"] <= line["ms_per_step"] * 1.001   # the decode call is part of the step
    e = line["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert "sm_mhz" in line["clocks"] and "reasons" in line["clocks"]
    # the compact targets are the line's last key
    assert list(line.keys())[-1] == "targets"
    t = line["targets"]
    for name in ("longctx_splitk", "gqa8b_prefix", "mha7b"):
        assert 0 < t[name]["frac"] < 1.2, name
        # each call after an L2 flush, between its own events: no faster than back to back
        assert 0 < t[name]["frac_l2_flushed"] <= t[name]["frac"] * 1.02, name


def test_bench_prefill_figures():
    """bench.py --prefill-only: the bench step's prefill figure, and a short chunk
    over a long cached context faster with its keys split than whole."""
    res = subprocess.run(
        [sys.executable, os.path.join(REPO, "bench.py"), "--prefill-only", "--prefill-reps", "5"],
        capture_output=True, text=True, timeout=900, cwd=REPO)
    assert res.returncode == 0, res.stderr[-3000:]
    pf = json.loads(res.stdout.strip().splitlines()[-1])["prefill"]
    assert 0 < pf["frac"] < 1.2
    c = pf["chunk128_after16k"]
    assert 0 < c["split_us"] < c["whole_us"]
