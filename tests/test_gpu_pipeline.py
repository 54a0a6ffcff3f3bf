"""Steps issued back to back, as the bench and a serving loop issue them (needs
a GPU).

* The bench's end-to-end loop (bench.time_e2e): every step copies its inputs
  from pinned host memory into one of two device staging buffers on a copy
  stream and reads its output back on that stream while the next step
  computes. Each step here gets its own queries, so a step that read a staging
  buffer still being refilled, or an output read back before its step wrote it
  (or after the step two later overwrote it), gives a row of the wrong step.
  Every read-back output is checked against the oracle.
* Two decode steps in a row through paged_kv_append_tokens, the second with
  sequences whose context is empty. The kernels are chained by programmatic
  dependent launch, so the second step's kernels may start while the first
  decode still runs; the empty sequences' zero rows must not be overwritten by
  the first decode's late writes of the same rows.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_233_gb300 as pk
from paged_support import TOL, oracle_fill, to_f64, to_np
from workloads import make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.load()
    torch.cuda.set_device(0)
    for opt in (pk.OPT_DECODE_PATH, pk.OPT_CTAS_PER_SM, pk.OPT_STAGES):
        pk.set_option(opt, 0)


@pytest.mark.parametrize("partition", [0, 64, -1])
def test_e2e_pipeline_outputs_match_oracle(orc, partition):
    import bench
    rng = np.random.default_rng(41)
    lens = rng.integers(1, 700, size=24)
    wl = make_workload("e2e", "f16", lens, 32, 32, 128, 16, 41)
    step = bench.Step(wl, torch.device("cuda", 0), partition)
    steps = 8
    gen = torch.Generator(device="cuda")
    gen.manual_seed(4242)
    qs = [torch.randn(step.t["q"].shape, generator=gen, device="cuda").to(torch.float16)
          for _ in range(5)]
    host_inputs = [bench.pack_host_inputs(bench.e2e_sources(step, q=q))[0] for q in qs]
    outputs = [torch.full(step.out.shape, float("nan"), dtype=step.out.dtype).pin_memory()
               for _ in range(steps)]
    pk.device_errors(reset=True)
    bench.time_e2e(step, steps, host_inputs=host_inputs, outputs=outputs)
    assert pk.device_errors() == 0
    okc, ovc, _ = oracle_fill(orc, wl, step.t)
    refs = [orc.decode(to_np(q), okc, ovc, wl.block_tables, wl.context_lens, wl.scale, wl.dtype)
            for q in qs]
    for i in range(steps):
        got = to_f64(outputs[i])
        err = float(np.abs(got - refs[i % len(qs)]).max())
        assert err <= TOL["f16"], f"step {i}: max-abs error {err:.3e}"
        # and it is not the output of the step's neighbour
        other = refs[(i + 1) % len(qs)]
        assert float(np.abs(got - other).max()) > 10 * TOL["f16"], f"step {i}: neighbour's row"


def test_empty_sequences_after_a_full_step_get_zero_rows(orc):
    """64 sequences (512 units of 4 kv heads: two rounds over the persistent
    grid, the last sequences in the second), decoded unsplit; then a step in
    which the last 8 sequences are empty (their tokens are padding, their
    lengths 0), decoded into the same output. Repeated so that the window in
    which the second decode could start early is met more than once."""
    S, Hq, Hkv, D, B = 64, 32, 32, 128, 16
    rng = np.random.default_rng(43)
    lens = rng.integers(900, 1100, size=S)
    wl = make_workload("pdl", "f16", lens, Hq, Hkv, D, B, 43)
    from workloads import materialize, new_pools
    t = materialize(wl, "cuda")
    kc, vc = new_pools(wl, "cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    fill_seq = torch.from_numpy(wl.fill_seq).cuda()
    fill_pos = torch.from_numpy(wl.fill_pos).cuda()
    pk.paged_kv_append_tokens(t["k_fill"], t["v_fill"], bt, fill_seq, fill_pos, kc, vc)
    step_seq = torch.from_numpy(wl.step_seq).cuda()
    pos_full = torch.from_numpy(wl.step_pos).cuda()
    empty = np.arange(S - 8, S)
    pos_empty = pos_full.clone()
    pos_empty[torch.from_numpy(empty).cuda()] = -1          # padding: nothing appended
    lens_full = torch.from_numpy(wl.context_lens).cuda()
    lens_empty = lens_full.clone()
    lens_empty[torch.from_numpy(empty).cuda()] = 0
    out = torch.empty_like(t["q"])
    pk.device_errors(reset=True)
    for _ in range(6):
        pk.paged_kv_append_tokens(t["k_step"], t["v_step"], bt, step_seq, pos_full, kc, vc)
        pk.paged_attention_decode(t["q"], kc, vc, bt, lens_full, wl.scale, out)
        pk.paged_kv_append_tokens(t["k_step"], t["v_step"], bt, step_seq, pos_empty, kc, vc)
        pk.paged_attention_decode(t["q"], kc, vc, bt, lens_empty, wl.scale, out)
    torch.cuda.synchronize()
    assert pk.device_errors() == 0
    got = to_f64(out)
    assert np.all(got[empty] == 0.0), "an empty sequence's row holds the previous step's values"
    okc, ovc, _ = oracle_fill(orc, wl, t)
    lens_e = wl.context_lens.copy()
    lens_e[empty] = 0
    ref = orc.decode(to_np(t["q"]), okc, ovc, wl.block_tables, lens_e, wl.scale, wl.dtype)
    err = float(np.abs(got - ref).max())
    assert err <= TOL["f16"], f"max-abs error {err:.3e}"
