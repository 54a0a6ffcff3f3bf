"""The hot path on streams other than the default one (needs a GPU).

Every entry point enqueues on the current torch stream, or on the stream it
is given, and returns without waiting. These tests run the whole step (slot
mapping, append, split-K decode with its merge, chunked prefill) under
``torch.cuda.stream(side)`` and with ``stream=`` on a second stream, behind a
torch kernel on the same stream that writes the inputs the library then
reads, and compare with the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_233_gb300 as pk
from paged_support import TOL, oracle_decode, oracle_fill, to_f64, to_np
from workloads import chunked_prefill, make_workload, materialize, new_pools, prefill_queries

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.load()
    torch.cuda.set_device(0)
    for opt in (pk.OPT_DECODE_PATH, pk.OPT_CTAS_PER_SM, pk.OPT_STAGES, pk.OPT_PREFILL_PATH):
        pk.set_option(opt, 0)


def run_step(wl, t, stream):
    """Pools, slots and a split-K decode, all enqueued on `stream` (None: the
    current stream). The step's q is first overwritten on the same stream by a
    torch copy from a scaled version, so a decode that ran on another stream
    could read it half-written."""
    kc, vc = new_pools(wl, "cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    lens = torch.from_numpy(wl.context_lens).cuda()
    for seq, pos, k, v in ((wl.fill_seq, wl.fill_pos, t["k_fill"], t["v_fill"]),
                           (wl.step_seq, wl.step_pos, t["k_step"], t["v_step"])):
        sm = torch.empty(len(seq), dtype=torch.int64, device="cuda")
        pk.paged_kv_slot_mapping(bt, torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda(), sm,
                                 wl.num_blocks, wl.block_size, stream=stream)
        pk.paged_kv_append(k, v, sm, kc, vc, stream=stream)
    q = torch.empty_like(t["q"])
    q.copy_(t["q"] * 0.5)   # on the current stream
    out = torch.full_like(q, float("nan"))
    ws = pk.new_workspace(q, bt, wl.block_size, 32)
    pk.paged_attention_decode(q, kc, vc, bt, lens, wl.scale, out, 32, ws, stream=stream)
    return kc, vc, q, out


@pytest.mark.parametrize("how", ["current", "explicit"])
def test_decode_step_on_a_side_stream(orc, how):
    wl = make_workload("streams", "f16", [1, 40, 77, 300, 1000], 8, 2, 128, 16, 31)
    t = materialize(wl, "cuda")
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        # for "explicit" the calls name the side stream while it is also current,
        # so the torch copy of q and the library's kernels share it either way
        kc, vc, q, out = run_step(wl, t, side if how == "explicit" else None)
    side.synchronize()
    assert pk.device_errors() == 0
    okc, ovc, _ = oracle_fill(orc, wl, t)
    assert to_np(kc).tobytes() == okc.tobytes() and to_np(vc).tobytes() == ovc.tobytes()
    ref = oracle_decode(orc, wl, q, okc, ovc)
    err = float(np.abs(to_f64(out) - ref).max())
    assert err <= TOL["f16"], err


def test_explicit_stream_differs_from_current(orc):
    """stream= wins over the current stream: the decode runs on `other` after
    an event that orders it behind the side stream's writes of q."""
    wl = make_workload("streams2", "bf16", [33, 600, 129], 8, 2, 64, 16, 32)
    t = materialize(wl, "cuda")
    torch.cuda.synchronize()
    side, other = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(side):
        kc, vc = new_pools(wl, "cuda")
        bt = torch.from_numpy(wl.block_tables).cuda()
        lens = torch.from_numpy(wl.context_lens).cuda()
        for seq, pos, k, v in ((wl.fill_seq, wl.fill_pos, t["k_fill"], t["v_fill"]),
                               (wl.step_seq, wl.step_pos, t["k_step"], t["v_step"])):
            sm = torch.empty(len(seq), dtype=torch.int64, device="cuda")
            pk.paged_kv_slot_mapping(bt, torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda(),
                                     sm, wl.num_blocks, wl.block_size)
            pk.paged_kv_append(k, v, sm, kc, vc)
        q = t["q"].clone()
        done = torch.cuda.Event()
        done.record(side)
        out = torch.full_like(q, float("nan"))
        ws = pk.new_workspace(q, bt, wl.block_size, 64)
        other.wait_event(done)
        pk.paged_attention_decode(q, kc, vc, bt, lens, wl.scale, out, 64, ws, stream=other)
    other.synchronize()
    side.synchronize()
    assert pk.device_errors() == 0
    okc, ovc, _ = oracle_fill(orc, wl, t)
    ref = oracle_decode(orc, wl, q, okc, ovc)
    err = float(np.abs(to_f64(out) - ref).max())
    assert err <= TOL["bf16"], err


def test_prefill_on_a_side_stream(orc):
    wl, qs = chunked_prefill("streams_prefill", "f16", [20, 0, 300], [50, 130, 17], 8, 2, 128, 16, 33)
    t = materialize(wl, "cuda")
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        kc, vc = new_pools(wl, "cuda")
        bt = torch.from_numpy(wl.block_tables).cuda()
        for seq, pos, k, v in ((wl.fill_seq, wl.fill_pos, t["k_fill"], t["v_fill"]),
                               (wl.step_seq, wl.step_pos, t["k_step"], t["v_step"])):
            sm = torch.empty(len(seq), dtype=torch.int64, device="cuda")
            pk.paged_kv_slot_mapping(bt, torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda(),
                                     sm, wl.num_blocks, wl.block_size)
            pk.paged_kv_append(k, v, sm, kc, vc)
        q = prefill_queries(wl, qs, "cuda")
        out = torch.full_like(q, float("nan"))
        pk.paged_attention_prefill(q, kc, vc, bt, torch.from_numpy(qs).cuda(),
                                   torch.from_numpy(wl.context_lens).cuda(), wl.scale, out, 130)
    side.synchronize()
    assert pk.device_errors() == 0
    okc, ovc, _ = oracle_fill(orc, wl, t)
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, wl.dtype)
    err = float(np.abs(to_f64(out) - ref).max())
    assert err <= TOL["f16"], err


def test_prefill_key_split_on_a_side_stream_and_in_a_graph(orc):
    """The key split (two kernels, the merge the programmatic dependent of the
    prefill kernel) on a side stream against the oracle, then captured in a
    CUDA graph: a replay on new queries equals an eager call on them, bit for
    bit."""
    wl, qs = chunked_prefill("streams_split", "f16", [2100, 0, 3300], [50, 130, 17], 8, 2, 128, 16, 34)
    t = materialize(wl, "cuda")
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        kc, vc = new_pools(wl, "cuda")
        bt = torch.from_numpy(wl.block_tables).cuda()
        for seq, pos, k, v in ((wl.fill_seq, wl.fill_pos, t["k_fill"], t["v_fill"]),
                               (wl.step_seq, wl.step_pos, t["k_step"], t["v_step"])):
            sm = torch.empty(len(seq), dtype=torch.int64, device="cuda")
            pk.paged_kv_slot_mapping(bt, torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda(),
                                     sm, wl.num_blocks, wl.block_size)
            pk.paged_kv_append(k, v, sm, kc, vc)
        q = prefill_queries(wl, qs, "cuda")
        qs_d = torch.from_numpy(qs).cuda()
        lens_d = torch.from_numpy(wl.context_lens).cuda()
        ws = pk.prefill_workspace(q)
        out = torch.full_like(q, float("nan"))
        pk.paged_attention_prefill(q, kc, vc, bt, qs_d, lens_d, wl.scale, out, 130, workspace=ws, key_parts=4)
    side.synchronize()
    assert pk.device_errors() == 0
    okc, ovc, _ = oracle_fill(orc, wl, t)
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, wl.dtype)
    assert float(np.abs(to_f64(out) - ref).max()) <= TOL["f16"]
    # captured once, replayed on new queries
    graph = torch.cuda.CUDAGraph()
    out_g = torch.full_like(q, float("nan"))
    with torch.cuda.graph(graph):
        pk.paged_attention_prefill(q, kc, vc, bt, qs_d, lens_d, wl.scale, out_g, 130, workspace=ws,
                                   key_parts=4)
    q.copy_(q.flip(0))
    graph.replay()
    out_e = torch.full_like(q, float("nan"))
    pk.paged_attention_prefill(q, kc, vc, bt, qs_d, lens_d, wl.scale, out_e, 130, workspace=ws, key_parts=4)
    torch.cuda.synchronize()
    assert pk.device_errors() == 0
    assert torch.equal(out_g, out_e)


def test_concurrent_host_threads(orc):
    """Two host threads decode at once, each on its own stream, with batches of
    different sizes through the same kernel instantiation: the launchers'
    per-device records (shared memory opened, occupancy of the last size asked
    about) are read and replaced by both threads while launches are in flight."""
    import threading

    cases = []
    for name, lens, seed in (("threads_a", [3, 70, 500, 17, 900], 34),
                             ("threads_b", [int(x) for x in np.linspace(1, 1200, 40)], 35)):
        wl = make_workload(name, "f16", lens, 8, 2, 128, 16, seed)
        t = materialize(wl, "cuda")
        kc, vc, q, _ = run_step(wl, t, None)
        cases.append((wl, t, kc, vc, q))
    torch.cuda.synchronize()
    results, errors = [None, None], []

    def worker(i):
        try:
            wl, _, kc, vc, q = cases[i]
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                bt = torch.from_numpy(wl.block_tables).cuda()
                lens = torch.from_numpy(wl.context_lens).cuda()
                ws = pk.new_workspace(q, bt, wl.block_size, 32)
                outs = []
                for rep in range(40):
                    out = torch.full_like(q, float("nan"))
                    pk.paged_attention_decode(q, kc, vc, bt, lens, wl.scale, out, 32 if rep % 2 else 0,
                                              ws)
                    outs.append(out)
            s.synchronize()
            results[i] = outs
        except Exception as e:   # surfaced by the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    assert pk.device_errors() == 0
    for i, (wl, t, kc, vc, q) in enumerate(cases):
        okc, ovc, _ = oracle_fill(orc, wl, t)
        ref = oracle_decode(orc, wl, q, okc, ovc)
        split = to_np(results[i][1]).tobytes()
        for rep, out in enumerate(results[i]):
            err = float(np.abs(to_f64(out) - ref).max())
            assert err <= TOL["f16"], (i, rep, err)
            if rep % 2:
                # the same split call gives the same bits every time
                assert to_np(out).tobytes() == split, (i, rep)
