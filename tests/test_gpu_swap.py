"""Block swap between device pools and pinned host pools, CUDA path against the
oracle (needs a GPU).

Swap-out and swap-in must leave both pools bit-exact to the oracle's (blocks
not named by a pair keep their bytes, out-of-pool ids are flagged and
skipped); a sequence swapped out and back into other blocks must decode
bit-identically; and the continuous-batching trace with swap preemption must
decode every (request, position) exactly as a run with nothing preempted.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_233_gb300 as pk
from oracle_pins import poison
from paged_support import gpu_decode, gpu_fill, to_np
from workloads import cb_trace, materialize, preset, step_inputs, trace_tensors

pytestmark = pytest.mark.gpu

TDT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.load()
    torch.cuda.set_device(0)
    for opt in (pk.OPT_DECODE_PATH, pk.OPT_CTAS_PER_SM, pk.OPT_STAGES):
        pk.set_option(opt, 0)


def pinned_pools(n, B, Hkv, D, dtype):
    k = torch.full((n, B, Hkv, D), float("nan"), dtype=TDT[dtype]).pin_memory()
    v = torch.full((n, B, Hkv, D), float("nan"), dtype=TDT[dtype]).pin_memory()
    return k, v


@pytest.mark.parametrize("dtype,B,Hkv,D", [("f16", 16, 32, 128), ("bf16", 8, 2, 64),
                                           ("f32", 32, 1, 64), ("bf16", 16, 8, 128)])
def test_swap_out_and_in_bit_exact(orc, dtype, B, Hkv, D):
    NB, NH = 48, 20
    g = torch.Generator(device="cuda").manual_seed(21)
    kc = torch.randn(NB, B, Hkv, D, generator=g, device="cuda").to(TDT[dtype])
    vc = torch.randn(NB, B, Hkv, D, generator=g, device="cuda").to(TDT[dtype])
    hk, hv = pinned_pools(NH, B, Hkv, D, dtype)
    okc, ovc = to_np(kc).copy(), to_np(vc).copy()
    ohk, ohv = poison(hk.shape, dtype), poison(hv.shape, dtype)
    rng = np.random.default_rng(22)
    out_pairs = np.stack([rng.choice(NB, 14, replace=False), rng.choice(NH, 14, replace=False)],
                         1).astype(np.int32)
    out_pairs[3, 0] = out_pairs[7, 0]                 # one source read twice
    pk.device_errors(reset=True)
    pk.paged_kv_swap_blocks(kc, vc, hk, hv, torch.from_numpy(out_pairs).cuda())
    torch.cuda.synchronize()
    assert pk.device_errors() == 0
    assert orc.swap_blocks(okc, ovc, ohk, ohv, out_pairs) == 0
    assert to_np(hk).tobytes() == ohk.tobytes() and to_np(hv).tobytes() == ohv.tobytes()
    assert to_np(kc).tobytes() == okc.tobytes() and to_np(vc).tobytes() == ovc.tobytes()
    # swap back in, into other device blocks
    in_pairs = np.stack([out_pairs[:, 1], rng.choice(NB, 14, replace=False)], 1).astype(np.int32)
    pk.paged_kv_swap_blocks(hk, hv, kc, vc, torch.from_numpy(in_pairs).cuda())
    assert pk.device_errors() == 0
    assert orc.swap_blocks(ohk, ohv, okc, ovc, in_pairs) == 0
    assert to_np(kc).tobytes() == okc.tobytes() and to_np(vc).tobytes() == ovc.tobytes()


def test_out_of_pool_ids_are_flagged_and_skipped(orc):
    B, Hkv, D, dtype = 16, 4, 64, "f16"
    kc = torch.randn(10, B, Hkv, D, device="cuda").half()
    vc = torch.randn(10, B, Hkv, D, device="cuda").half()
    hk, hv = pinned_pools(4, B, Hkv, D, dtype)
    ohk, ohv = poison(hk.shape, dtype), poison(hv.shape, dtype)
    # 9 is a device block but not a host block; 10 and -1 are neither
    pairs = np.array([[2, 1], [9, 9], [10, 0], [-1, 2], [5, 3]], np.int32)
    pk.device_errors(reset=True)
    pk.paged_kv_swap_blocks(kc, vc, hk, hv, torch.from_numpy(pairs).cuda())
    assert pk.device_errors() & 0x02
    assert orc.swap_blocks(to_np(kc), to_np(vc), ohk, ohv, pairs) == 3
    assert to_np(hk).tobytes() == ohk.tobytes() and to_np(hv).tobytes() == ohv.tobytes()


def test_device_pools_of_different_sizes_and_pinned_pairs(orc):
    B, Hkv, D, dtype = 8, 8, 128, "bf16"
    a_k = torch.randn(30, B, Hkv, D, device="cuda").bfloat16()
    a_v = torch.randn(30, B, Hkv, D, device="cuda").bfloat16()
    b_k = torch.zeros(12, B, Hkv, D, device="cuda").bfloat16()
    b_v = torch.zeros(12, B, Hkv, D, device="cuda").bfloat16()
    ob_k, ob_v = to_np(b_k).copy(), to_np(b_v).copy()
    pairs = np.array([[29, 0], [0, 11], [13, 5], [13, 6]], np.int32)
    host_pairs = torch.from_numpy(pairs).pin_memory()     # the kernel reads the pairs in place
    pk.paged_kv_swap_blocks(a_k, a_v, b_k, b_v, host_pairs)
    torch.cuda.synchronize()
    assert orc.swap_blocks(to_np(a_k), to_np(a_v), ob_k, ob_v, pairs) == 0
    assert to_np(b_k).tobytes() == ob_k.tobytes() and to_np(b_v).tobytes() == ob_v.tobytes()
    assert pk.device_errors() == 0


def test_zero_pairs_and_pageable_memory():
    kc = torch.zeros(4, 16, 2, 64, device="cuda").half()
    pk.paged_kv_swap_blocks(kc, kc, kc, kc, torch.zeros(0, 2, dtype=torch.int32, device="cuda"))
    # the C entry point itself refuses pageable host memory before launching anything
    lib = pk.load()
    host = torch.zeros(4, 16, 2, 64).half()
    pairs = torch.zeros(1, 2, dtype=torch.int32, device="cuda")
    vp = ctypes.c_void_p
    st = lib.paged_kv_swap_blocks(vp(kc.data_ptr()), vp(kc.data_ptr()), 4, vp(host.data_ptr()),
                                  vp(host.data_ptr()), 4, vp(pairs.data_ptr()), 1, 16, 2, 64, 1,
                                  vp(torch.cuda.current_stream().cuda_stream))
    assert st == -1
    assert pk.device_errors() == 0


def test_swapped_sequences_decode_bit_identically():
    """Llama-2-7B-shaped workload (64 sequences, fp16): swap out a quarter of
    the sequences' blocks to pinned host memory, overwrite those device blocks,
    swap them back into other free blocks and rewrite the tables."""
    wl = preset("mha7b")
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    before, _ = gpu_decode(wl, t["q"], kc, vc, bt, 320)
    tables = wl.block_tables.copy()
    used = set(tables[tables >= 0].tolist())
    free = [b for b in range(wl.num_blocks) if b not in used]
    rng = np.random.default_rng(23)
    victims, moved = [], 0
    for s in rng.permutation(wl.num_seqs):
        n = int((tables[s] >= 0).sum())
        if moved + n > len(free):
            continue
        victims.append(int(s))
        moved += n
        if len(victims) == wl.num_seqs // 4:
            break
    assert victims
    src = np.concatenate([tables[s][tables[s] >= 0] for s in victims]).astype(np.int32)
    hk, hv = pinned_pools(len(src), wl.block_size, wl.n_kv_heads, wl.head_dim, wl.dtype)
    host_ids = np.arange(len(src), dtype=np.int32)
    pk.paged_kv_swap_blocks(kc, vc, hk, hv, torch.from_numpy(np.stack([src, host_ids], 1)).cuda())
    idx = torch.from_numpy(src.astype(np.int64)).cuda()
    kc[idx] = float("nan")                                # the freed blocks are reused
    vc[idx] = float("nan")
    dst = np.asarray(free[:len(src)], np.int32)
    pk.paged_kv_swap_blocks(hk, hv, kc, vc, torch.from_numpy(np.stack([host_ids, dst], 1)).cuda())
    k = 0
    for s in victims:
        n = int((tables[s] >= 0).sum())
        tables[s, :n] = dst[k:k + n]
        k += n
    after, _ = gpu_decode(wl, t["q"], kc, vc, torch.from_numpy(tables).cuda(), 320)
    assert pk.device_errors() == 0
    assert torch.equal(before.view(torch.int16), after.view(torch.int16))


def run_trace_swap(tw, tensors, P, host_blocks):
    """Every step of a trace on the GPU, swaps included; decoded rows by (rid, position)."""
    shape = (tw.num_blocks, tw.block_size, tw.n_kv_heads, tw.head_dim)
    kc = torch.full(shape, float("nan"), dtype=tw.torch_dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    hk = torch.full((host_blocks,) + shape[1:], float("nan"), dtype=tw.torch_dtype).pin_memory()
    hv = torch.full_like(hk, float("nan")).pin_memory()
    rows = {}
    for plan in tw.plans:
        if len(plan.swap_in):
            pk.paged_kv_swap_blocks(hk, hv, kc, vc, torch.from_numpy(plan.swap_in).cuda())
        if len(plan.swap_out):
            pk.paged_kv_swap_blocks(kc, vc, hk, hv, torch.from_numpy(plan.swap_out).cuda())
        x = step_inputs(tw, plan, tensors, "cuda")
        slots = torch.empty(len(plan.token_row), dtype=torch.int64, device="cuda")
        pk.paged_kv_slot_mapping(x["block_tables"], x["token_row"], x["token_pos"], slots,
                                 tw.num_blocks, tw.block_size)
        pk.paged_kv_append(x["k"], x["v"], slots, kc, vc)
        out = torch.empty_like(x["q"])
        ws = pk.new_workspace(x["q"], x["block_tables"], tw.block_size, P)
        pk.paged_attention_decode(x["q"], kc, vc, x["block_tables"], x["context_lens"], tw.scale,
                                  out, P, ws)
        got = out.double().cpu().numpy()
        for b, rid in enumerate(plan.rids):
            rows[(rid, int(plan.query_pos[b]))] = got[b]
    assert pk.device_errors() == 0
    return rows


def test_trace_with_swap_preemption_changes_no_output():
    small = cb_trace(block_size=16, slots=32, pool_tokens=2048, preempt="swap",
                     host_tokens=16384)
    large = cb_trace(block_size=16, slots=32, pool_tokens=65536)
    assert small.preemptions > 0 and large.preemptions == 0
    assert sum(len(p.swap_out) for p in small.plans) > 0
    tensors = trace_tensors(small, "cuda")
    got_small = run_trace_swap(small, tensors, 256, 16384 // 16)
    got_large = run_trace_swap(large, tensors, 256, 1)
    assert got_small.keys() == got_large.keys()
    for key in got_small:
        assert np.array_equal(got_small[key], got_large[key]), key
