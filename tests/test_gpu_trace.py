"""The continuous-batching workload, step by step, CUDA path against the fp64
oracle (needs a GPU).

Each step's slot mapping must be bit-exact, each step's decode within the
dtype's tolerance on every output, and the pools bit-exact at the end. The
run with a small pool (LIFO preemption by recompute) must decode every
(request, position) exactly as the run with a pool large enough that nothing
is preempted.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_233_gb300 as pk
from oracle_pins import poison
from paged_support import TOL, to_f64, to_np
from workloads import cb_trace, step_inputs, trace_tensors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.load()
    torch.cuda.set_device(0)
    for opt in (pk.OPT_DECODE_PATH, pk.OPT_CTAS_PER_SM, pk.OPT_STAGES):
        pk.set_option(opt, 0)


def run_trace(tw, tensors, P, orc=None):
    """Run every step on the GPU (and on the oracle when given). Returns
    {(rid, query position): decoded row as float64} and the final GPU pools."""
    shape = (tw.num_blocks, tw.block_size, tw.n_kv_heads, tw.head_dim)
    kc = torch.full(shape, float("nan"), dtype=tw.torch_dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    if orc is not None:
        okc, ovc = poison(shape, tw.dtype), poison(shape, tw.dtype)
    rows = {}
    for plan in tw.plans:
        x = step_inputs(tw, plan, tensors, "cuda")
        T = len(plan.token_row)
        slots = torch.empty(T, dtype=torch.int64, device="cuda")
        pk.paged_kv_slot_mapping(x["block_tables"], x["token_row"], x["token_pos"], slots,
                                 tw.num_blocks, tw.block_size)
        pk.paged_kv_append(x["k"], x["v"], slots, kc, vc)
        out = torch.empty_like(x["q"])
        ws = pk.new_workspace(x["q"], x["block_tables"], tw.block_size, P)
        pk.paged_attention_decode(x["q"], kc, vc, x["block_tables"], x["context_lens"], tw.scale,
                                  out, P, ws)
        got = to_f64(out)
        if orc is not None:
            sm = orc.slot_mapping(plan.block_tables, plan.token_row, plan.token_pos, tw.block_size)
            assert np.array_equal(slots.cpu().numpy(), sm), f"step {plan.step}: slots differ"
            assert orc.append(to_np(x["k"]), to_np(x["v"]), sm, okc, ovc) == 0
            ref = orc.decode(to_np(x["q"]), okc, ovc, plan.block_tables, plan.context_lens,
                             tw.scale, tw.dtype)
            err = float(np.abs(got - ref).max())
            assert err <= TOL[tw.dtype], f"step {plan.step}: max-abs error {err:.3e}"
        for b, rid in enumerate(plan.rids):
            rows[(rid, int(plan.query_pos[b]))] = got[b]
    if orc is not None:
        assert to_np(kc).view(np.uint8).tobytes() == okc.view(np.uint8).tobytes()
        assert to_np(vc).view(np.uint8).tobytes() == ovc.view(np.uint8).tobytes()
    assert pk.device_errors() == 0
    return rows


@pytest.mark.parametrize("block_size", [8, 16, 32])
def test_trace_matches_oracle(orc, block_size):
    tw = cb_trace(block_size=block_size, slots=64)
    tensors = trace_tensors(tw, "cuda")
    rows = run_trace(tw, tensors, 256, orc)
    assert len(rows) == sum(r.output_len for r in tw.requests)


def test_preemption_by_recompute_changes_no_output(orc):
    small = cb_trace(block_size=16, slots=32, pool_tokens=2048)
    large = cb_trace(block_size=16, slots=32, pool_tokens=65536)
    assert small.preemptions > 0 and large.preemptions == 0
    tensors = trace_tensors(small, "cuda")
    got_small = run_trace(small, tensors, 256, orc)
    got_large = run_trace(large, tensors, 256)
    assert got_small.keys() == got_large.keys()
    for key in got_small:
        assert np.array_equal(got_small[key], got_large[key]), key
