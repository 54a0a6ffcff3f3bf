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


SLOTS = [8, 16, 32, 64, 128, 256]


@pytest.mark.parametrize("slots", SLOTS)
@pytest.mark.parametrize("block_size", [8, 16, 32])
def test_trace_matches_oracle(orc, block_size, slots):
    """Separate slot-mapping and append calls, 256-token partitions."""
    tw = cb_trace(block_size=block_size, slots=slots)
    tensors = trace_tensors(tw, "cuda")
    rows = run_trace(tw, tensors, 256, orc)
    assert len(rows) == sum(r.output_len for r in tw.requests)
    assert max(len(p.rids) for p in tw.plans) <= slots


def oracle_trace(orc, tw, tensors):
    """Every step's decoded rows and the final pools, all on the oracle."""
    shape = (tw.num_blocks, tw.block_size, tw.n_kv_heads, tw.head_dim)
    okc, ovc = poison(shape, tw.dtype), poison(shape, tw.dtype)
    refs, slots = [], []
    for plan in tw.plans:
        x = step_inputs(tw, plan, tensors, "cpu")
        sm = orc.slot_mapping(plan.block_tables, plan.token_row, plan.token_pos, tw.block_size)
        assert orc.append(to_np(x["k"]), to_np(x["v"]), sm, okc, ovc) == 0
        refs.append(orc.decode(to_np(x["q"]), okc, ovc, plan.block_tables, plan.context_lens,
                               tw.scale, tw.dtype))
        slots.append(sm)
    return refs, slots, okc, ovc


def bench_launches_against_oracle(orc, tw):
    """The bench's launches: one paged_kv_append_tokens (slots written out too)
    and one balanced-split decode per step, one workspace for every step."""
    tensors = trace_tensors(tw, "cuda")
    refs, ref_slots, okc, ovc = oracle_trace(orc, tw, {k: v.cpu() for k, v in tensors.items()})
    shape = (tw.num_blocks, tw.block_size, tw.n_kv_heads, tw.head_dim)
    kc = torch.full(shape, float("nan"), dtype=tw.torch_dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    P = pk.PARTITION_BALANCED
    ws_bytes = max(pk.paged_attention_workspace_bytes(len(p.rids), tw.n_q_heads, tw.head_dim,
                                                      p.block_tables.shape[1], tw.block_size, P)
                   for p in tw.plans)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    pk.device_errors(reset=True)
    for i, plan in enumerate(tw.plans):
        x = step_inputs(tw, plan, tensors, "cuda")
        sm = torch.empty(len(plan.token_row), dtype=torch.int64, device="cuda")
        pk.paged_kv_append_tokens(x["k"], x["v"], x["block_tables"], x["token_row"],
                                  x["token_pos"], kc, vc, slot_mapping=sm)
        out = torch.full_like(x["q"], float("nan"))
        pk.paged_attention_decode(x["q"], kc, vc, x["block_tables"], x["context_lens"], tw.scale,
                                  out, P, ws)
        assert np.array_equal(sm.cpu().numpy(), ref_slots[i]), f"step {plan.step}: slots differ"
        err = float(np.abs(to_f64(out) - refs[i]).max())
        assert err <= TOL[tw.dtype], f"step {plan.step}: max-abs error {err:.3e}"
    assert to_np(kc).view(np.uint8).tobytes() == okc.view(np.uint8).tobytes()
    assert to_np(vc).view(np.uint8).tobytes() == ovc.view(np.uint8).tobytes()
    assert pk.device_errors() == 0


@pytest.mark.parametrize("slots", SLOTS)
@pytest.mark.parametrize("block_size", [8, 16, 32])
def test_trace_bench_launches_match_oracle(orc, block_size, slots):
    bench_launches_against_oracle(orc, cb_trace(block_size=block_size, slots=slots))


def test_trace_bench_launches_with_preemption_match_oracle(orc):
    """The bench's reduced-pool trace (4,096 token slots, 64 slots): LIFO
    preemption by recompute re-appends the victims' tokens inside the steps."""
    tw = cb_trace(block_size=16, slots=64, pool_tokens=4096)
    assert tw.preemptions > 0
    bench_launches_against_oracle(orc, tw)


@pytest.mark.parametrize("block_size,slots", [(16, 8), (16, 64), (8, 32), (32, 16)])
def test_trace_graph_replay_matches_oracle(orc, block_size, slots):
    """The bench's graph-issued trace: the whole pass captured once in a CUDA
    graph; after two replays every step's output and the pools equal the
    oracle's (appends rewrite the same bytes, so replays are idempotent)."""
    import bench
    tw = cb_trace(block_size=block_size, slots=slots)
    shape = (tw.num_blocks, tw.block_size, tw.n_kv_heads, tw.head_dim)
    pools = (torch.full(shape, float("nan"), dtype=tw.torch_dtype, device="cuda"),
             torch.full(shape, float("nan"), dtype=tw.torch_dtype, device="cuda"))
    tr = bench.TraceRun(tw, "cuda", pk.PARTITION_BALANCED, pools=pools)
    pk.device_errors(reset=True)
    tr.run_pass()
    torch.cuda.synchronize()
    for _, x in tr.steps:
        x["out"].fill_(float("nan"))
    g = tr.capture()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    refs, _, okc, ovc = oracle_trace(orc, tw, {k: v.cpu() for k, v in trace_tensors(tw, "cuda").items()})
    for i, (plan, x) in enumerate(tr.steps):
        err = float(np.abs(to_f64(x["out"]) - refs[i]).max())
        assert err <= TOL[tw.dtype], f"step {plan.step}: max-abs error {err:.3e}"
    assert to_np(tr.kc).view(np.uint8).tobytes() == okc.view(np.uint8).tobytes()
    assert to_np(tr.vc).view(np.uint8).tobytes() == ovc.view(np.uint8).tobytes()
    assert pk.device_errors() == 0


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
