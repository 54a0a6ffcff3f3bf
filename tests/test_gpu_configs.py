"""The named workloads at full size, in the launch configuration bench.py
times, against the fp64 oracle (needs a GPU).

The whole pools must be bit-exact to the oracle's; the decode output is
checked element by element on a sample of (sequence, kv head) units that the
oracle computes one by one (the longest and shortest sequences, members of a
shared-prefix group, and seeded random picks), and split-K is checked against
the unsplit decode on every output.
"""
import numpy as np
import pytest
import torch

import bench
import paged_kv_cache_233_gb300 as pk
from paged_support import (assert_close, gpu_decode, gpu_fill, oracle_decode, oracle_fill, to_f64,
                           to_np, units_to_rows, TOL)
from workloads import materialize, preset

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.load()
    torch.cuda.set_device(0)
    for opt in (pk.OPT_DECODE_PATH, pk.OPT_CTAS_PER_SM, pk.OPT_STAGES):
        pk.set_option(opt, 0)


def sample_units(wl, n_random=8, seed=0):
    rng = np.random.default_rng(seed)
    lens = wl.context_lens
    seqs = {int(np.argmax(lens)), int(np.argmin(lens))}
    for grp in wl.groups[:1]:
        seqs.update(grp[:2])
    seqs.update(int(s) for s in rng.choice(wl.num_seqs, size=min(n_random, wl.num_seqs), replace=False))
    units = []
    for s in sorted(seqs):
        for h in sorted({0, wl.n_kv_heads - 1, int(rng.integers(wl.n_kv_heads))}):
            units.append((s, h))
    return units


@pytest.mark.parametrize("name", ["mha7b", "gqa8b_prefix", "longctx_splitk"])
def test_full_size_workload(orc, name):
    wl = preset(name)
    P = bench.PARTITION[name]
    t = materialize(wl, "cuda")
    kc, vc, bt, slots = gpu_fill(wl, t)
    pk.device_errors(reset=True)
    out, _ = gpu_decode(wl, t["q"], kc, vc, bt, P)
    torch.cuda.synchronize()
    assert pk.device_errors() == 0
    okc, ovc, oslots = oracle_fill(orc, wl, t)
    for tag in ("fill", "step"):
        assert np.array_equal(slots[tag].cpu().numpy(), oslots[tag])
    assert to_np(kc).tobytes() == okc.tobytes()
    assert to_np(vc).tobytes() == ovc.tobytes()
    del okc
    units = sample_units(wl)
    ref = oracle_decode(orc, wl, t["q"], to_np(kc), ovc, units=units)
    err = assert_close(out, ref, wl.dtype, rows=units_to_rows(wl, units), what=name)
    # split-K (bench configuration) against one pass per (sequence, kv head), on every output
    whole, _ = gpu_decode(wl, t["q"], kc, vc, bt, 0)
    diff = float(np.abs(to_f64(out) - to_f64(whole)).max())
    assert diff <= TOL[wl.dtype], (name, diff)
    print(f"{name}: {len(units)} units, max-abs error vs oracle {err:.2e}, split vs whole {diff:.2e}")
