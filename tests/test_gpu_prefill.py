"""Chunked-prefill attention, CUDA path against the fp64 oracle (needs a GPU).

The chunk's K/V go into NaN-poisoned pools through the library's slot mapping
and append, as a serving step would do; then every query row of the chunk
must match the oracle's causal attention over its sequence within the dtype's
tolerance, on both kernels (warp-level MMA and tcgen05). A prompt prefilled
chunk by chunk must give bit-identical rows to one pass over the whole prompt; one-row chunks must agree with decode; bad
lengths are flagged on the device error word and leave their rows untouched.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_233_gb300 as pk
from paged_support import TOL, gpu_fill, oracle_fill, to_f64, to_np
from workloads import chunked_prefill, materialize, prefill_mha7b, prefill_queries

pytestmark = pytest.mark.gpu

# (tokens cached before the chunk, chunk length): empty and one-row chunks, a
# chunk that is the whole prompt, ragged tails around 64-key and 64-row tiles
CASES = [(0, 1), (0, 77), (13, 50), (100, 130), (300, 1), (37, 0), (64, 64), (5, 200)]


@pytest.fixture(scope="module", autouse=True, params=[1, 2], ids=["mma_sync", "tcgen05"])
def path(request):
    """Every test runs on both kernels: warp-level MMA (1) and tcgen05 (2)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.load()
    torch.cuda.set_device(0)
    pk.device_errors(reset=True)
    pk.set_option(pk.OPT_PREFILL_PATH, request.param)
    yield request.param
    pk.set_option(pk.OPT_PREFILL_PATH, 0)


def build(dtype, D, B, g, seed, cases=CASES, n_kv=2):
    before = [c[0] for c in cases]
    chunk = [c[1] for c in cases]
    wl, qs = chunked_prefill("prefill_case", dtype, before, chunk, g * n_kv, n_kv, D, B, seed)
    tensors = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, tensors)
    q = prefill_queries(wl, qs, "cuda")
    return wl, qs, tensors, q, kc, vc, bt


def prefill(wl, qs, q, kc, vc, bt, lens=None, max_query_len=None):
    out = torch.full_like(q, float("nan"))
    lens = wl.context_lens if lens is None else lens
    pk.paged_attention_prefill(q, kc, vc, bt, torch.from_numpy(np.asarray(qs, np.int32)).cuda(),
                               torch.from_numpy(np.asarray(lens, np.int32)).cuda(), wl.scale, out,
                               max_query_len)
    return out


@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("B", [8, 16, 32])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_matches_oracle(orc, dtype, D, B, g):
    wl, qs, tensors, q, kc, vc, bt = build(dtype, D, B, g, seed=100 + D + B + g)
    out = prefill(wl, qs, q, kc, vc, bt)
    assert pk.device_errors() == 0
    okc, ovc, _ = oracle_fill(orc, wl, tensors)
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, dtype)
    got = to_f64(out)
    assert not np.isnan(got).any()
    err = float(np.abs(got - ref).max())
    assert err <= TOL[dtype], f"max-abs error {err:.3e}"


@pytest.mark.parametrize("g", [3, 5, 6, 7, 16, 48, 64])
def test_prefill_odd_and_large_groups(orc, g):
    """Groups that do not divide a tile's rows (the warp-level kernel's 64, the
    tcgen05 kernel's 128: its Q tiles then hold 128 // g whole tokens, 96 rows
    for 48), and a whole tile of heads."""
    cases = [(0, 9), (40, 33), (7, 70)]
    wl, qs, tensors, q, kc, vc, bt = build("bf16", 64, 16, g, seed=200 + g, cases=cases, n_kv=1)
    out = prefill(wl, qs, q, kc, vc, bt)
    assert pk.device_errors() == 0
    okc, ovc, _ = oracle_fill(orc, wl, tensors)
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, "bf16")
    assert float(np.abs(to_f64(out) - ref).max()) <= TOL["bf16"]


@pytest.mark.parametrize("dtype,B", [("f16", 16), ("bf16", 8)])
def test_chunk_by_chunk_equals_one_pass(dtype, B):
    """The prompts' rows come out bit-identical whether a call covers the whole
    prompt or the prompt is prefilled in chunks over several calls."""
    chunks = [[128, 128, 45], [1, 100, 49], [64, 1, 1]]
    prompts = [sum(c) for c in chunks]
    wl, qs, tensors, q, kc, vc, bt = build(dtype, 128, B, 4, seed=300,
                                           cases=[(0, n) for n in prompts])
    whole = prefill(wl, qs, q, kc, vc, bt)
    done = [0] * len(prompts)
    for r in range(3):
        sizes = [c[r] for c in chunks]
        cqs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
        lens = np.array([done[s] + sizes[s] for s in range(len(prompts))], np.int32)
        rows = torch.cat([q[qs[s] + done[s]:qs[s] + lens[s]] for s in range(len(prompts))])
        part = prefill(wl, cqs, rows.contiguous(), kc, vc, bt, lens=lens)
        for s in range(len(prompts)):
            a = part[cqs[s]:cqs[s + 1]]
            b = whole[qs[s] + done[s]:qs[s] + lens[s]]
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (r, s)
            done[s] = int(lens[s])
    assert pk.device_errors() == 0


def test_one_row_chunks_agree_with_decode(orc):
    wl, qs, tensors, q, kc, vc, bt = build("f16", 128, 16, 4, seed=400,
                                           cases=[(0, 1), (16, 1), (170, 1), (999, 1)])
    out = prefill(wl, qs, q, kc, vc, bt)
    dec = torch.full_like(q, float("nan"))
    pk.paged_attention_decode(q, kc, vc, bt, torch.from_numpy(wl.context_lens).cuda(), wl.scale,
                              dec, 0, None)
    okc, ovc, _ = oracle_fill(orc, wl, tensors)
    ref = orc.decode(to_np(q), okc, ovc, wl.block_tables, wl.context_lens, wl.scale, "f16")
    assert float(np.abs(to_f64(out) - ref).max()) <= TOL["f16"]
    assert float(np.abs(to_f64(dec) - ref).max()) <= TOL["f16"]
    assert pk.device_errors() == 0


def test_bad_lengths_are_flagged_and_left_unwritten(orc):
    cases = [(10, 20), (5, 30), (0, 300)]
    wl, qs, tensors, q, kc, vc, bt = build("bf16", 64, 16, 2, seed=500, cases=cases)
    # sequence 1 claims fewer cached tokens than its chunk has rows
    lens = wl.context_lens.copy()
    lens[1] = 29
    pk.device_errors(reset=True)
    out = prefill(wl, qs, q, kc, vc, bt, lens=lens)
    assert pk.device_errors() & 0x04
    got = to_f64(out)
    assert np.isnan(got[qs[1]:qs[2]]).all()
    okc, ovc, _ = oracle_fill(orc, wl, tensors)
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, "bf16",
                      units=[(0, 0), (0, 1), (2, 0), (2, 1)])
    keep = np.r_[qs[0]:qs[1], qs[2]:qs[3]]
    assert float(np.abs(got[keep] - ref[keep]).max()) <= TOL["bf16"]
    # a chunk longer than the grid that max_query_len sized (300 rows; a CTA
    # covers at most 128 tokens of group 2 on either kernel)
    out = prefill(wl, qs, q, kc, vc, bt, max_query_len=10)
    assert pk.device_errors() & 0x08
    assert np.isnan(to_f64(out)[qs[2]:qs[3]]).all()
    assert pk.device_errors() == 0


def test_fp32_and_unsupported_shapes_are_refused():
    q = torch.zeros(4, 4, 64, device="cuda")
    kc = torch.zeros(8, 16, 2, 64, device="cuda")
    bt = torch.zeros(1, 8, dtype=torch.int32, device="cuda")
    qs = torch.tensor([0, 4], dtype=torch.int32, device="cuda")
    lens = torch.tensor([4], dtype=torch.int32, device="cuda")
    with pytest.raises(pk.PagedKVError, match="unsupported"):
        pk.paged_attention_prefill(q, kc, kc, bt, qs, lens, 0.125, torch.empty_like(q))
    q16 = torch.zeros(4, 4, 96, device="cuda").half()
    kc16 = torch.zeros(8, 16, 2, 96, device="cuda").half()
    with pytest.raises(pk.PagedKVError, match="unsupported"):
        pk.paged_attention_prefill(q16, kc16, kc16, bt, qs, lens, 0.125, torch.empty_like(q16))
    assert pk.device_errors() == 0


def test_prefill_full_size_sampled(orc):
    """The bench's chunked-prefill step at full size (Llama-2-7B layer, 16
    sequences appending 512-token chunks after up to 3584 cached tokens),
    sampled (sequence, head) units against the oracle."""
    wl, qs = prefill_mha7b()
    tensors = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, tensors)
    q = prefill_queries(wl, qs, "cuda")
    out = prefill(wl, qs, q, kc, vc, bt, max_query_len=512)
    assert pk.device_errors() == 0
    got = to_f64(out)
    assert not np.isnan(got).any()
    rng = np.random.default_rng(6)
    units = [(int(s), int(h)) for s, h in zip(rng.choice(wl.num_seqs, 4, replace=False),
                                              rng.choice(wl.n_kv_heads, 4, replace=False))]
    # the oracle attends over its own pools (its slot mapping + append of the
    # same tokens), and the GPU's pools equal them byte for byte
    okc, ovc, _ = oracle_fill(orc, wl, tensors)
    assert to_np(kc).view(np.uint8).tobytes() == okc.view(np.uint8).tobytes()
    assert to_np(vc).view(np.uint8).tobytes() == ovc.view(np.uint8).tobytes()
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, "f16",
                      units=units)
    for s, h in units:
        err = float(np.abs(got[qs[s]:qs[s + 1], h] - ref[qs[s]:qs[s + 1], h]).max())
        assert err <= TOL["f16"], (s, h, err)


@pytest.mark.parametrize("g,n_kv", [(1, 8), (3, 4), (8, 4)])
def test_many_items_per_cta(orc, g, n_kv):
    """Far more (sequence, query tile, kv head) items than SMs, so that the
    tcgen05 kernel's persistent CTAs each work through many: chunks of one
    row to three query tiles, chunks whose second Q tile is empty, contexts
    on a 64-key boundary and ragged ones, every output row against the oracle
    (groups that divide 128, and 3, whose Q tiles hold 42 whole tokens, 126
    rows)."""
    rng = np.random.default_rng(520)
    before = rng.integers(0, 900, size=40)
    chunk = rng.integers(1, 600, size=40)
    before[:4] = [0, 64, 128, 0]          # contexts ending on a 64-key boundary
    chunk[:4] = [64, 64, 128, 100]
    cases = list(zip(before.tolist(), chunk.tolist()))
    wl, qs, tensors, q, kc, vc, bt = build("bf16", 64, 16, g, seed=521 + g, cases=cases, n_kv=n_kv)
    pk.device_errors(reset=True)
    out = prefill(wl, qs, q, kc, vc, bt)
    assert pk.device_errors() == 0
    okc, ovc, _ = oracle_fill(orc, wl, tensors)
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, "bf16")
    err = float(np.abs(to_f64(out) - ref).max())
    assert err <= TOL["bf16"], err


def test_more_sequences_than_the_ranking_holds_with_a_bad_one(orc):
    """300 sequences (the tcgen05 kernel ranks at most 256 by length and
    keeps the given order beyond that), one of them with a length shorter
    than its chunk: it is flagged and left unwritten, every other row matches
    the oracle."""
    rng = np.random.default_rng(530)
    cases = list(zip(rng.integers(0, 200, size=300).tolist(), rng.integers(1, 40, size=300).tolist()))
    wl, qs, tensors, q, kc, vc, bt = build("f16", 64, 16, 2, seed=531, cases=cases, n_kv=2)
    lens = wl.context_lens.copy()
    bad = 150
    lens[bad] = int(qs[bad + 1] - qs[bad]) - 1
    pk.device_errors(reset=True)
    out = prefill(wl, qs, q, kc, vc, bt, lens=lens)
    assert pk.device_errors() == 0x04
    got = to_f64(out)
    assert np.isnan(got[qs[bad]:qs[bad + 1]]).all()
    okc, ovc, _ = oracle_fill(orc, wl, tensors)
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, "f16")
    keep = np.r_[0:qs[bad], qs[bad + 1]:qs[-1]]
    err = float(np.abs(got[keep] - ref[keep]).max())
    assert err <= TOL["f16"], err


@pytest.mark.parametrize("g", [1, 8])
def test_query_rows_past_every_chunk_stay_out(orc, g):
    """q holds 50 NaN rows after the last chunk (num_tokens past the chunks'
    end): a Q tile that reaches past its chunk reads them (or the next
    sequence's rows), and none of it may reach a chunk's output row; the
    output rows past the chunks stay as they were."""
    cases = [(10, 30), (0, 77), (200, 100), (5, 3)]
    wl, qs, tensors, q, kc, vc, bt = build("f16", 128, 16, g, seed=540 + g, cases=cases, n_kv=2)
    pad = torch.full((50,) + tuple(q.shape[1:]), float("nan"), dtype=q.dtype, device=q.device)
    qp = torch.cat([q, pad])
    out = torch.full_like(qp, float("nan"))
    out[q.shape[0]:] = 7.0
    pk.device_errors(reset=True)
    pk.paged_attention_prefill(qp, kc, vc, bt, torch.from_numpy(np.asarray(qs, np.int32)).cuda(),
                               torch.from_numpy(np.asarray(wl.context_lens, np.int32)).cuda(),
                               wl.scale, out)
    assert pk.device_errors() == 0
    assert bool((out[q.shape[0]:] == 7.0).all())
    okc, ovc, _ = oracle_fill(orc, wl, tensors)
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, "f16")
    got = to_f64(out[:q.shape[0]])
    assert not np.isnan(got).any()
    assert float(np.abs(got - ref).max()) <= TOL["f16"]


def prefill_split(wl, qs, q, kc, vc, bt, parts, lens=None, workspace=None, out=None):
    out = torch.full_like(q, float("nan")) if out is None else out
    lens = wl.context_lens if lens is None else lens
    ws = pk.prefill_workspace(q) if workspace is None else workspace
    pk.paged_attention_prefill(q, kc, vc, bt, torch.from_numpy(np.asarray(qs, np.int32)).cuda(),
                               torch.from_numpy(np.asarray(lens, np.int32)).cuda(), wl.scale, out,
                               workspace=ws, key_parts=parts)
    return out


# long cached contexts (items of 33 to 72 key tiles, split in up to 5 parts of
# 8 to 16 key tiles) beside short ones (not split) in one call
SPLIT_CASES = [(0, 1), (1100, 1), (2500, 77), (1024, 50), (3000, 130), (37, 0), (1984, 64),
               (4300, 200)]


@pytest.mark.parametrize("parts", [2, 3, 32])
@pytest.mark.parametrize("g", [1, 3, 8])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_key_split_matches_oracle(orc, dtype, D, g, parts):
    """The call's key tiles in equal ranges over the SMs, no item in more than
    2, 3 or 32 of them (a piece can lie past a Q tile's rows, a range can hold
    the end of one item and the start of the next, short items whole), the
    pieces' states merged: every row against the oracle."""
    wl, qs, tensors, q, kc, vc, bt = build(dtype, D, 16, g, seed=600 + D + g + parts, cases=SPLIT_CASES)
    pk.device_errors(reset=True)
    out = prefill_split(wl, qs, q, kc, vc, bt, parts)
    assert pk.device_errors() == 0
    okc, ovc, _ = oracle_fill(orc, wl, tensors)
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, dtype)
    got = to_f64(out)
    assert not np.isnan(got).any()
    err = float(np.abs(got - ref).max())
    assert err <= TOL[dtype], f"max-abs error {err:.3e}"


@pytest.mark.parametrize("g", [16, 64])
def test_key_split_large_groups(orc, g):
    """The key split at groups of 16 and 64 (Q tiles of 8 and 2 whole tokens):
    long and short contexts in one call against the oracle."""
    cases = [(2000, 9), (0, 33), (3100, 70), (1500, 1)]
    wl, qs, tensors, q, kc, vc, bt = build("bf16", 64, 16, g, seed=670 + g, cases=cases, n_kv=1)
    pk.device_errors(reset=True)
    out = prefill_split(wl, qs, q, kc, vc, bt, 4)
    assert pk.device_errors() == 0
    okc, ovc, _ = oracle_fill(orc, wl, tensors)
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, "bf16")
    assert float(np.abs(to_f64(out) - ref).max()) <= TOL["bf16"]


def test_key_split_without_a_workspace_takes_one_from_torch(orc):
    """The binding allocates the split's workspace when the caller passes none."""
    cases = [(3000, 100)]
    wl, qs, tensors, q, kc, vc, bt = build("f16", 64, 16, 1, seed=660, cases=cases, n_kv=4)
    out = torch.full_like(q, float("nan"))
    pk.paged_attention_prefill(q, kc, vc, bt, torch.from_numpy(np.asarray(qs, np.int32)).cuda(),
                               torch.from_numpy(np.asarray(wl.context_lens, np.int32)).cuda(), wl.scale,
                               out, key_parts=0)
    okc, ovc, _ = oracle_fill(orc, wl, tensors)
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, "f16")
    assert float(np.abs(to_f64(out) - ref).max()) <= TOL["f16"]


def test_key_split_automatic_parts_and_a_short_workspace(orc, path):
    """key_parts 0 splits a call of fewer items than SMs; a workspace smaller
    than the split needs is refused (on the tcgen05 kernel: the warp-level MMA
    kernel does not split, and needs none); the workspace's size follows the
    SM count alone."""
    cases = [(1920, 128)]   # one sequence, one 128-token chunk after 1920 cached tokens
    wl, qs, tensors, q, kc, vc, bt = build("f16", 128, 16, 1, seed=640, cases=cases, n_kv=32)
    out = prefill_split(wl, qs, q, kc, vc, bt, 0)
    okc, ovc, _ = oracle_fill(orc, wl, tensors)
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, "f16")
    assert float(np.abs(to_f64(out) - ref).max()) <= TOL["f16"]
    sms = torch.cuda.get_device_properties(q.device).multi_processor_count

    def r256(x):
        return (x + 255) // 256 * 256

    rows = 2 * sms * 256
    assert pk.prefill_workspace_bytes(128) == r256(500 * 4) + r256(rows * 128 * 4) + 2 * r256(rows * 4)
    assert pk.prefill_workspace_bytes(96) == 0
    short = torch.empty(pk.prefill_workspace_bytes(q.shape[2]) - 256, dtype=torch.uint8, device=q.device)
    if path == 2:
        with pytest.raises(pk.PagedKVError):
            prefill_split(wl, qs, q, kc, vc, bt, 4, workspace=short)
    else:
        out = prefill_split(wl, qs, q, kc, vc, bt, 4, workspace=short)
        assert float(np.abs(to_f64(out) - ref).max()) <= TOL["f16"]


def test_key_split_of_many_items_and_past_its_item_limit(orc):
    """Near the split's 500-item limit (ranges of short items end to end, a
    long item cut) and past it (whole items at any key_parts): the oracle."""
    rng = np.random.default_rng(680)
    for n_seq, n_kv in ((60, 8), (62, 8), (63, 8)):   # 480 and 496 items split; 504 run whole
        cases = [(int(b), int(c)) for b, c in zip(rng.integers(0, 300, n_seq), rng.integers(1, 200, n_seq))]
        cases[0] = (5000, 200)
        wl, qs, tensors, q, kc, vc, bt = build("bf16", 64, 16, 1, seed=680 + n_seq, cases=cases, n_kv=n_kv)
        pk.device_errors(reset=True)
        out = prefill_split(wl, qs, q, kc, vc, bt, 32)
        assert pk.device_errors() == 0
        okc, ovc, _ = oracle_fill(orc, wl, tensors)
        ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, "bf16")
        assert float(np.abs(to_f64(out) - ref).max()) <= TOL["bf16"], (n_seq, n_kv)


@pytest.mark.parametrize("D", [64, 128])
def test_key_split_one_long_item_among_many_short(orc, D):
    """20 items (more than SMs / 9: the merge loads 8 pieces at a time), two of
    them over a 30,000-token context cut into about 30 ranges, so that the
    merge takes several round trips per row; the short ones whole: the oracle."""
    cases = [(30000, 40)] + [(0, 10)] * 9
    wl, qs, tensors, q, kc, vc, bt = build("bf16", D, 16, 1, seed=690 + D, cases=cases, n_kv=2)
    pk.device_errors(reset=True)
    out = prefill_split(wl, qs, q, kc, vc, bt, 32)
    assert pk.device_errors() == 0
    okc, ovc, _ = oracle_fill(orc, wl, tensors)
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, "bf16")
    got = to_f64(out)
    assert not np.isnan(got).any()
    assert float(np.abs(got - ref).max()) <= TOL["bf16"]


def test_key_split_leaves_flagged_and_padding_rows_alone(orc):
    """Under a key split a sequence whose length is shorter than its chunk is
    flagged and its rows left unwritten, and output rows past the chunks keep
    what they held, as without the split."""
    cases = [(2100, 30), (0, 77), (3000, 100), (5, 3)]
    wl, qs, tensors, q, kc, vc, bt = build("bf16", 128, 16, 2, seed=650, cases=cases, n_kv=2)
    pad = torch.zeros((20,) + tuple(q.shape[1:]), dtype=q.dtype, device=q.device)
    qp = torch.cat([q, pad])
    out = torch.full_like(qp, float("nan"))
    out[q.shape[0]:] = 7.0
    lens = wl.context_lens.copy()
    bad = 2
    lens[bad] = int(qs[bad + 1] - qs[bad]) - 1
    pk.device_errors(reset=True)
    prefill_split(wl, qs, qp, kc, vc, bt, 3, lens=lens, out=out)
    assert pk.device_errors() == 0x04
    assert bool((out[q.shape[0]:] == 7.0).all())
    got = to_f64(out[:q.shape[0]])
    assert np.isnan(got[qs[bad]:qs[bad + 1]]).all()
    okc, ovc, _ = oracle_fill(orc, wl, tensors)
    ref = orc.prefill(to_np(q), okc, ovc, wl.block_tables, qs, wl.context_lens, wl.scale, "bf16")
    keep = np.r_[0:qs[bad], qs[bad + 1]:qs[-1]]
    assert float(np.abs(got[keep] - ref[keep]).max()) <= TOL["bf16"]
