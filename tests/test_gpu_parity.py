"""CUDA path against the fp64 oracle, element by element (needs a GPU).

Append and slot mapping must be bit-exact; decode must be within max-abs
2e-3 (fp16), 1.5e-2 (bf16) or 1e-5 (fp32) of the oracle.
"""
import math
import zlib

import numpy as np
import pytest
import torch

import paged_kv_cache_233_gb300 as pk
from paged_support import (TOL, assert_close, gpu_decode, gpu_fill, oracle_decode, oracle_fill,
                           to_f64, to_np, units_to_rows)
from workloads import make_workload, materialize, preset

pytestmark = pytest.mark.gpu

PATHS = {"auto": 0, "simt": 1, "mma": 2}


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.load()
    torch.cuda.set_device(0)
    yield
    pk.set_option(pk.OPT_DECODE_PATH, 0)


@pytest.fixture(autouse=True)
def clean_error_word():
    pk.device_errors(reset=True)
    yield
    pk.set_option(pk.OPT_DECODE_PATH, 0)


def run_both(orc, wl, partition_tokens=0, path="auto"):
    t = materialize(wl, "cuda")
    kc, vc, bt, slots = gpu_fill(wl, t)
    pk.set_option(pk.OPT_DECODE_PATH, PATHS[path])
    out, ws = gpu_decode(wl, t["q"], kc, vc, bt, partition_tokens)
    okc, ovc, oslots = oracle_fill(orc, wl, t)
    ref = oracle_decode(orc, wl, t["q"], okc, ovc)
    return dict(t=t, kc=kc, vc=vc, bt=bt, slots=slots, out=out, ws=ws, okc=okc, ovc=ovc,
                oslots=oslots, ref=ref)


# ---------------------------------------------------------------------------
# The tiny workload, end to end
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("partition_tokens", [0, 16, 32, -1])
def test_tiny_workload(orc, partition_tokens):
    wl = preset("tiny")
    r = run_both(orc, wl, partition_tokens)
    for tag in ("fill", "step"):
        assert np.array_equal(r["slots"][tag].cpu().numpy(), r["oslots"][tag])
    assert to_np(r["kc"]).tobytes() == r["okc"].tobytes()
    assert to_np(r["vc"]).tobytes() == r["ovc"].tobytes()
    assert_close(r["out"], r["ref"], "f32", what="tiny")
    assert pk.device_errors() == 0


def test_tiny_workload_lengths_before_the_append(orc):
    """The other reading of the tiny workload's lengths: decode over the tokens
    held before the step's append (the new token is in the pool but unread)."""
    wl = preset("tiny")
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    okc, ovc, _ = oracle_fill(orc, wl, t)
    wl.context_lens = wl.context_lens - 1
    out, _ = gpu_decode(wl, t["q"], kc, vc, bt)
    assert_close(out, oracle_decode(orc, wl, t["q"], okc, ovc), "f32", what="tiny-before")


# ---------------------------------------------------------------------------
# Sweeps over the supported shapes, both decode paths, split and not
# ---------------------------------------------------------------------------

SWEEP_LENS = [1, 2, 7, 8, 9, 15, 16, 17, 31, 33, 49, 64, 67, 100, 203, 517]


def sweep_cases():
    for dtype in ("f32", "f16", "bf16"):
        for D in (64, 128):
            for B in (8, 16, 32):
                for g in (1, 2, 4, 8):
                    paths = ["simt"] if dtype == "f32" else ["simt", "mma"]
                    for path in paths:
                        for P in (0, 48, -1):
                            yield pytest.param(dtype, D, B, g, path, P,
                                               id=f"{dtype}-D{D}-B{B}-g{g}-{path}-P{P}")


@pytest.mark.parametrize("dtype,D,B,g,path,P", list(sweep_cases()))
def test_decode_sweep(orc, dtype, D, B, g, path, P):
    Hkv = 2
    seed = zlib.crc32(f"{dtype}-{D}-{B}-{g}".encode()) % 10000
    wl = make_workload("sweep", dtype, SWEEP_LENS, Hkv * g, Hkv, D, B, seed, pool_factor=1.5)
    r = run_both(orc, wl, P, path)
    assert pk.last_decode_path() == PATHS[path]
    assert to_np(r["kc"]).tobytes() == r["okc"].tobytes()
    assert to_np(r["vc"]).tobytes() == r["ovc"].tobytes()
    assert_close(r["out"], r["ref"], dtype, what=f"{dtype} D{D} B{B} g{g} {path} P{P}")
    assert pk.device_errors() == 0


@pytest.mark.parametrize("dtype,g,want", [("f16", 1, "mma"), ("bf16", 2, "mma"), ("f16", 8, "mma"),
                                          ("f32", 1, "simt"), ("f32", 4, "simt")])
def test_automatic_path_choice(orc, dtype, g, want):
    """The automatic decode path takes the tensor-core consumer for every
    16-bit pool (it measured faster at every group size) and the CUDA-core
    consumer for fp32; either way the result matches the oracle."""
    wl = make_workload("auto", dtype, [5, 40, 130], 2 * g, 2, 64, 16, 61)
    r = run_both(orc, wl, 0, "auto")
    assert pk.last_decode_path() == PATHS[want]
    assert_close(r["out"], r["ref"], dtype, what=f"auto path {dtype} g{g}")
    assert pk.device_errors() == 0


@pytest.mark.parametrize("dtype,path", [("bf16", "mma"), ("f16", "simt"), ("f32", "simt")])
def test_split_partition_states(orc, dtype, path):
    """The split-K partition states in the workspace match the oracle's
    per-partition (m, l, o) for every (sequence, head, partition)."""
    P, D, Hkv, g = 32, 64, 2, 4
    wl = make_workload("parts", dtype, [5, 32, 33, 97, 130], Hkv * g, Hkv, D, 16, 77)
    r = run_both(orc, wl, P, path)
    S, Hq = wl.num_seqs, wl.n_q_heads
    max_parts = -(-(wl.max_blocks_per_seq * wl.block_size) // P)
    rows = S * Hq * max_parts
    r256 = lambda x: (x + 255) // 256 * 256
    ws = r["ws"].cpu().numpy().view(np.float32)
    o_all = ws[:rows * D].reshape(S, Hq, max_parts, D)
    m_all = ws[r256(rows * D * 4) // 4:][:rows].reshape(S, Hq, max_parts)
    l_all = ws[(r256(rows * D * 4) + r256(rows * 4)) // 4:][:rows].reshape(S, Hq, max_parts)
    q = to_np(r["t"]["q"])
    checked = 0
    for s, L in enumerate(wl.context_lens):
        nparts = -(-int(L) // P)
        if nparts < 2:
            continue
        for qh in range(Hq):
            for p_ in range(nparts):
                o, m, l = orc.decode_partition(q, r["okc"], r["ovc"], wl.block_tables, wl.scale,
                                               dtype, s, qh, p_ * P, min(int(L), (p_ + 1) * P))
                gm, gl, go = float(m_all[s, qh, p_]), float(l_all[s, qh, p_]), o_all[s, qh, p_]
                assert abs(gm - m) < 1e-4, (s, qh, p_, gm, m)
                assert abs(gl / math.exp(m - gm) - l) / l < 1e-4
                assert np.abs(go / gl - o / l).max() < TOL[dtype]
                checked += 1
    assert checked > 0
    assert_close(r["out"], r["ref"], dtype, what="split")


# ---------------------------------------------------------------------------
# Edge cases
# ---------------------------------------------------------------------------

def test_largest_batch_and_one_past_it(orc):
    """The largest batch the decode accepts (4096 sequences; their per-sequence
    unit counts live in shared memory), split and not, against sampled oracle
    rows; one sequence more is refused on the host."""
    rng = np.random.default_rng(44)
    lens = rng.integers(1, 80, size=4096)
    wl = make_workload("max_batch", "f16", lens, 4, 2, 64, 16, 45)
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    okc, ovc, _ = oracle_fill(orc, wl, t)
    units = [(int(s), int(h)) for s in rng.choice(wl.num_seqs, 24, replace=False) for h in range(2)]
    ref = oracle_decode(orc, wl, t["q"], okc, ovc, units=units)
    for P in (0, 32):
        out, _ = gpu_decode(wl, t["q"], kc, vc, bt, P)
        assert_close(out, ref, "f16", rows=units_to_rows(wl, units), what=f"P={P}")
    assert pk.device_errors() == 0
    q = torch.zeros(4097, 4, 64, dtype=torch.float16, device="cuda")
    bt2 = torch.zeros(4097, 1, dtype=torch.int32, device="cuda")
    lens2 = torch.ones(4097, dtype=torch.int32, device="cuda")
    with pytest.raises(pk.PagedKVError, match="unsupported"):
        pk.paged_attention_decode(q, kc, vc, bt2, lens2, wl.scale, torch.empty_like(q), 0, None)


def test_empty_and_single_token_contexts(orc):
    wl = make_workload("edge", "bf16", [1, 1, 16, 1], 8, 2, 128, 16, 5)
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    okc, ovc, _ = oracle_fill(orc, wl, t)
    wl.context_lens = np.array([0, 1, 16, 0], dtype=np.int32)
    for path in ("simt", "mma"):
        pk.set_option(pk.OPT_DECODE_PATH, PATHS[path])
        for P in (0, 16, -1):
            out, _ = gpu_decode(wl, t["q"], kc, vc, bt, P)
            o = to_f64(out)
            assert (o[0] == 0).all() and (o[3] == 0).all()
            assert_close(out, oracle_decode(orc, wl, t["q"], okc, ovc), "bf16", what="edge")
    assert pk.device_errors() == 0


def hpu4_cases():
    for dtype in ("f32", "f16", "bf16"):
        for D in (64, 128):
            for B in (8, 16, 32):
                for g in (1, 4, 8):
                    for P in (48, 256, -1, 16):
                        yield pytest.param(dtype, D, B, g, P,
                                           id=f"{dtype}-D{D}-B{B}-g{g}-P{P}")


@pytest.mark.parametrize("dtype,D,B,g,P", list(hpu4_cases()))
def test_split_with_four_kv_heads_per_unit(orc, dtype, D, B, g, P):
    """Four kv heads per unit (one consumer warp each, no cross-warp merge):
    partitions of 48 or 256 tokens (at most 32 per row, the row-per-warp merge
    kernel), 16-token partitions (rows of up to 69 partitions, the
    CTA-per-row merge kernel) and the balanced split; ragged lengths with
    empty contexts, called twice in a row on one workspace whose bytes start
    as 0xff, against the oracle."""
    Hkv = 4
    lens = SWEEP_LENS + [0, 1100, 0, 640]
    seed = zlib.crc32(f"hpu4-{dtype}-{D}-{B}-{g}".encode()) % 10000
    wl = make_workload("hpu4", dtype, lens, Hkv * g, Hkv, D, B, seed, pool_factor=1.5)
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    okc, ovc, _ = oracle_fill(orc, wl, t)
    ref = oracle_decode(orc, wl, t["q"], okc, ovc)
    lens_d = torch.from_numpy(wl.context_lens).cuda()
    ws = pk.new_workspace(t["q"], bt, wl.block_size, P)
    ws.fill_(255)
    for _ in range(2):
        out = torch.full_like(t["q"], float("nan"))
        pk.paged_attention_decode(t["q"], kc, vc, bt, lens_d, wl.scale, out, P, ws)
        assert_close(out, ref, dtype, what=f"{dtype} D{D} B{B} g{g} P{P}")
    assert pk.device_errors() == 0


@pytest.mark.parametrize("ctas", [1, 2, 8])
def test_balanced_split_over_skewed_lengths(orc, ctas):
    """Balanced shares cut single sequences into many pieces (one very long
    sequence among short ones, and more CTAs than tiles for the short ones)."""
    pk.set_option(pk.OPT_CTAS_PER_SM, ctas)
    try:
        for dtype, g in (("bf16", 8), ("f16", 1), ("f32", 2)):
            wl = make_workload("skew", dtype, [4000, 1, 17, 2, 33, 0 + 5], 4 * g, 4, 64, 16, 91)
            r = run_both(orc, wl, -1)
            assert_close(r["out"], r["ref"], dtype, what=f"balanced {dtype} ctas={ctas}")
        tiny = make_workload("few", "f16", [3, 20], 8, 4, 128, 16, 92)
        r = run_both(orc, tiny, -1)
        assert_close(r["out"], r["ref"], "f16", what="fewer tiles than CTAs")
    finally:
        pk.set_option(pk.OPT_CTAS_PER_SM, 0)
    assert pk.device_errors() == 0


# (name, dtype, q heads, kv heads, lengths low/high, sequences). K/V per token
# is 4 KiB for 8 kv heads x 128 (bf16) and 16 KiB for 32 x 128 (fp16), so every
# case's block tables can hold several times the L2's 126 MB: the ring holds
# three stages. The first two have short mean contexts (all three stages run),
# the last a mean of about 9,500 tokens (each CTA runs two of the three).
STAGE_RING_CASES = [
    ("three_stages_gqa", "bf16", 32, 8, (700, 1400), 48),
    ("three_stages_mha", "f16", 32, 32, (300, 900), 16),
    ("two_of_three_long", "bf16", 64, 8, (7000, 12000), 6),
]


@pytest.mark.parametrize("name,dtype,Hq,Hkv,lo_hi,S", STAGE_RING_CASES)
def test_balanced_split_stage_rings(orc, name, dtype, Hq, Hkv, lo_hi, S):
    """The balanced split's automatic stage ring, sized on the host from the
    block tables' width and chosen per CTA from the mean context, against the
    oracle on every output."""
    rng = np.random.default_rng(97)
    lens = rng.integers(lo_hi[0], lo_hi[1], size=S)
    wl = make_workload(name, dtype, lens, Hq, Hkv, 128, 16, 97)
    token_bytes = 2 * Hkv * 128 * 2
    assert S * wl.block_tables.shape[1] * 16 * token_bytes > 129e6   # more than the L2: three stages
    r = run_both(orc, wl, -1)
    assert_close(r["out"], r["ref"], dtype, what=f"balanced split, {name}")
    assert pk.device_errors() == 0


@pytest.mark.parametrize("ctas", [1, 8])
def test_balanced_split_ignores_stale_workspace(orc, ctas):
    """The balanced merge reads only the pieces the decode wrote: a workspace
    full of NaN bytes (every share's slots, including those of CTAs that got no
    tiles, which lie inside a long sequence's range of shares at 8 CTAs per SM)
    gives the same result as the oracle."""
    pk.set_option(pk.OPT_CTAS_PER_SM, ctas)
    try:
        for dtype, g, lens in (("f16", 1, [4000, 1, 17, 2, 33, 5]), ("bf16", 4, [3, 700, 20, 1, 64])):
            wl = make_workload("stale", dtype, lens, 4 * g, 4, 128, 16, 93)
            t = materialize(wl, "cuda")
            kc, vc, bt, _ = gpu_fill(wl, t)
            lens_d = torch.from_numpy(wl.context_lens).cuda()
            ws = pk.new_workspace(t["q"], bt, wl.block_size, pk.PARTITION_BALANCED)
            ws.fill_(255)
            out = torch.full_like(t["q"], float("nan"))
            pk.paged_attention_decode(t["q"], kc, vc, bt, lens_d, wl.scale, out, pk.PARTITION_BALANCED, ws)
            okc, ovc, _ = oracle_fill(orc, wl, t)
            assert_close(out, oracle_decode(orc, wl, t["q"], okc, ovc), dtype, what=f"stale {dtype} ctas={ctas}")
    finally:
        pk.set_option(pk.OPT_CTAS_PER_SM, 0)
    assert pk.device_errors() == 0


def test_empty_batch_is_a_no_op():
    q = torch.empty(0, 4, 64, device="cuda", dtype=torch.float16)
    kc = torch.zeros(4, 16, 2, 64, device="cuda", dtype=torch.float16)
    bt = torch.zeros(0, 2, dtype=torch.int32, device="cuda")
    lens = torch.zeros(0, dtype=torch.int32, device="cuda")
    pk.paged_attention_decode(q, kc, kc, bt, lens, 0.125, q.clone())
    torch.cuda.synchronize()


def test_bad_block_ids_and_lengths_are_flagged_not_dereferenced():
    wl = make_workload("bad", "f16", [40, 40], 4, 2, 64, 16, 3)
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    assert pk.device_errors() == 0
    bad = bt.clone()
    bad[0, 1] = wl.num_blocks + 1000          # past the pool
    bad[1, 0] = -7
    out, _ = gpu_decode(wl, t["q"], kc, vc, bad)
    assert pk.device_errors() & 0x02
    lens = torch.tensor([40, 10 ** 6], dtype=torch.int32, device="cuda")
    out = torch.empty_like(t["q"])
    pk.paged_attention_decode(t["q"], kc, vc, bt, lens, wl.scale, out)
    assert pk.device_errors() & 0x04


def test_slot_mapping_padding_and_errors(orc):
    wl = make_workload("slots", "f32", [20, 3], 2, 2, 64, 8, 9)
    bt = torch.from_numpy(wl.block_tables).cuda()
    seq = torch.tensor([0, 0, 1, 1, 5, 0], dtype=torch.int32, device="cuda")
    pos = torch.tensor([0, 19, 2, -1, 0, 10 ** 5], dtype=torch.int32, device="cuda")
    sm = torch.empty(6, dtype=torch.int64, device="cuda")
    pk.paged_kv_slot_mapping(bt, seq, pos, sm, wl.num_blocks, wl.block_size)
    got = sm.cpu().numpy()
    assert got[3] == -1 and got[4] == -1 and got[5] == -1
    ref = orc.slot_mapping(wl.block_tables, [0, 0, 1], [0, 19, 2], wl.block_size)
    assert got[:3].tolist() == ref.tolist()
    flags = pk.device_errors()
    assert flags & 0x10 and flags & 0x08


def test_append_skips_padding_and_flags_out_of_range_slots(orc):
    NB, B, Hkv, D = 4, 8, 2, 64
    kc = torch.full((NB, B, Hkv, D), float("nan"), device="cuda")
    vc = kc.clone()
    k = torch.randn(5, Hkv, D, device="cuda")
    v = torch.randn(5, Hkv, D, device="cuda")
    slots = torch.tensor([3, -1, NB * B, 31, 0], dtype=torch.int64, device="cuda")
    pk.paged_kv_append(k, v, slots, kc, vc)
    assert pk.device_errors() & 0x01
    okc = np.full((NB, B, Hkv, D), np.nan, np.float32)
    ovc = okc.copy()
    bad = orc.append(to_np(k), to_np(v), slots.cpu().numpy(), okc, ovc)
    assert bad == 1
    assert to_np(kc).tobytes() == okc.tobytes() and to_np(vc).tobytes() == ovc.tobytes()
