"""Pins that tie the fp64 oracle to something other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with:

* a library routine computing the same thing another way (numpy's float16,
  torch's bfloat16, numpy/scipy softmax attention on contiguous K/V),
* the pages' printed worked example of a block table,
* an invariant of the definition (block-id permutation, shared vs private
  prefix blocks, split-context identity),
* a closed-form special case (one token, identical keys, empty context).

The same functions run against deliberately broken builds of the oracle in
``test_oracle_mutants.py``; every mutant must trip at least one of them.
"""
import math
import os

import numpy as np
import scipy.special
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

STORAGE_NP = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}
NAN_BITS_BF16 = 0x7FC0


# ---------------------------------------------------------------------------
# Helpers that build small paged inputs (no oracle code involved).
# ---------------------------------------------------------------------------

def to_storage(x, dtype):
    """fp64/fp32 array -> stored elements (bf16 as uint16 bit patterns)."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float32))
    if dtype == "f32":
        return t.numpy().astype(np.float32)
    if dtype == "f16":
        return t.to(torch.float16).numpy()
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def widen_lib(a, dtype):
    """Stored elements -> float64 by the libraries' own conversions."""
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    return a.astype(np.float64)


def poison(shape, dtype):
    if dtype == "bf16":
        return np.full(shape, NAN_BITS_BF16, dtype=np.uint16)
    return np.full(shape, np.nan, dtype=STORAGE_NP[dtype])


def paged_case(seed, lens, B, Hq, Hkv, D, dtype, spare_blocks=3):
    """Random per-sequence contiguous K/V placed block by block in a shuffled pool.

    Block j of sequence s holds that sequence's tokens jB .. jB+B-1 (the
    pages' picture of a block: B consecutive tokens' keys and values).
    Returns the stored arrays and the contiguous fp64 copies.
    """
    rng = np.random.default_rng(seed)
    S = len(lens)
    need = [-(-L // B) for L in lens]
    NB = sum(need) + spare_blocks
    perm = rng.permutation(NB)
    MB = max(max(need), 1)
    bt = np.full((S, MB), -1, dtype=np.int32)
    k = 0
    for s in range(S):
        for j in range(need[s]):
            bt[s, j] = perm[k]
            k += 1
    kpool = poison((NB, B, Hkv, D), dtype)
    vpool = poison((NB, B, Hkv, D), dtype)
    Kc, Vc = [], []
    for s, L in enumerate(lens):
        Ks = to_storage(rng.standard_normal((L, Hkv, D)), dtype)
        Vs = to_storage(rng.standard_normal((L, Hkv, D)), dtype)
        for j in range(need[s]):
            n = min(B, L - j * B)
            kpool[bt[s, j], :n] = Ks[j * B:j * B + n]
            vpool[bt[s, j], :n] = Vs[j * B:j * B + n]
        Kc.append(widen_lib(Ks, dtype))
        Vc.append(widen_lib(Vs, dtype))
    q = to_storage(rng.standard_normal((S, Hq, D)), dtype)
    return dict(q=q, k=kpool, v=vpool, bt=bt, lens=np.asarray(lens, np.int32), Kc=Kc, Vc=Vc,
                qc=widen_lib(q, dtype), B=B, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype, NB=NB,
                scale=1.0 / math.sqrt(D))


def brute_force(case):
    """Contiguous softmax attention with numpy/scipy (query head h -> kv head h // g)."""
    S, Hq, D = case["q"].shape
    g = Hq // case["Hkv"]
    out = np.zeros((S, Hq, D))
    for s in range(S):
        if case["lens"][s] == 0:
            continue
        for h in range(Hq):
            K = case["Kc"][s][:, h // g, :]
            V = case["Vc"][s][:, h // g, :]
            z = case["scale"] * (K @ case["qc"][s, h])
            out[s, h] = scipy.special.softmax(z) @ V
    return out


def run_decode(orc, case, **kw):
    return orc.decode(case["q"], case["k"], case["v"], case["bt"], case["lens"], case["scale"],
                      case["dtype"], **kw)


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------------------
# Element decoding.
# ---------------------------------------------------------------------------

def pin_f16_decoding(orc):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_to_double(b) for b in bits.tolist()])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), f"fp16 decoding differs at {np.nonzero(~same)[0][:5]}"


def pin_bf16_decoding(orc):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = widen_lib(bits, "bf16")
    got = np.array([orc.bf16_to_double(b) for b in bits.tolist()])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), f"bf16 decoding differs at {np.nonzero(~same)[0][:5]}"


# ---------------------------------------------------------------------------
# Address translation.
# ---------------------------------------------------------------------------

def pin_block_table_example(orc):
    """The pages' printed 10-token, B = 4 sequence in blocks [5, 2, 9], grown to 13."""
    rows = read_golden("block_table_b4.txt")
    B = int(rows[0][1])
    n0, nblocks, waste = int(rows[1][1]), int(rows[1][3]), int(rows[1][5])
    table = [int(x) for x in rows[1][7:]]
    assert len(table) == nblocks
    bt = np.array([table], dtype=np.int32)
    held = [orc.slot(bt, 0, i, B) // B for i in range(n0)]
    assert held == sorted(held, key=table.index), "tokens leave logical block order"
    assert sorted(set(held), key=table.index) == table, "tokens not spread over the table"
    assert nblocks * B - n0 == waste
    for row in rows[2:]:
        n_tokens = int(row[2])
        grown = [int(x) for x in row[4:row.index("wrote")]]
        bt = np.array([grown], dtype=np.int32)
        pos = n_tokens - 1
        slot = orc.slot(bt, 0, pos, B)
        if row[-1] == "current":
            assert slot // B == table[-1] and slot % B != 0, (row, slot)
        else:
            assert slot // B == grown[-1] and slot % B == 0, (row, slot)
        table = grown


def pin_slot_bijection(orc):
    """Disjoint tables: every (seq, pos) gets its own slot, each block holds
    at most B consecutive positions, blocks are used in table order."""
    case = paged_case(11, [1, 5, 8, 13, 31], 8, 2, 1, 8, "f32")
    B, bt, lens = case["B"], case["bt"], case["lens"]
    seen = set()
    for s, L in enumerate(lens):
        slots = [orc.slot(bt, s, i, B) for i in range(L)]
        assert all(0 <= x < case["NB"] * B for x in slots)
        seen.update(slots)
        blocks = [x // B for x in slots]
        offs = [x % B for x in slots]
        assert offs == [i % B for i in range(L)]
        assert blocks == [int(bt[s, i // B]) for i in range(L)]
        assert len(set(blocks)) == -(-L // B)
    assert len(seen) == int(lens.sum())
    # the mapping entry point agrees with the single-slot function and pads with -1
    ts = np.array([0, 3, 4, 4, 2], np.int32)
    tp = np.array([0, 12, 30, -1, 7], np.int32)
    sm = orc.slot_mapping(bt, ts, tp, B)
    assert sm.tolist() == [orc.slot(bt, 0, 0, B), orc.slot(bt, 3, 12, B),
                           orc.slot(bt, 4, 30, B), -1, orc.slot(bt, 2, 7, B)]


def pin_append_scatter(orc):
    """Append writes each token row at its slot and leaves everything else alone."""
    rng = np.random.default_rng(5)
    NB, B, Hkv, D = 6, 4, 2, 8
    for dtype in ("f32", "f16", "bf16"):
        kpool = poison((NB, B, Hkv, D), dtype)
        vpool = poison((NB, B, Hkv, D), dtype)
        T = 9
        k = to_storage(rng.standard_normal((T, Hkv, D)), dtype)
        v = to_storage(rng.standard_normal((T, Hkv, D)), dtype)
        slots = rng.permutation(NB * B)[:T].astype(np.int64)
        slots[3] = -1
        slots[7] = NB * B + 2
        ek, ev = kpool.copy(), vpool.copy()
        keep = (slots >= 0) & (slots < NB * B)
        ek.reshape(NB * B, Hkv, D)[slots[keep]] = k[keep]
        ev.reshape(NB * B, Hkv, D)[slots[keep]] = v[keep]
        bad = orc.append(k, v, slots, kpool, vpool)
        assert bad == 1
        assert kpool.tobytes() == ek.tobytes() and vpool.tobytes() == ev.tobytes()


def pin_copy_blocks(orc):
    """Block copy equals numpy whole-block assignment; bad ids are skipped."""
    rng = np.random.default_rng(8)
    NB, B, Hkv, D = 7, 4, 2, 8
    for dtype in ("f32", "bf16"):
        k = to_storage(rng.standard_normal((NB, B, Hkv, D)), dtype)
        v = to_storage(rng.standard_normal((NB, B, Hkv, D)), dtype)
        pairs = np.array([[1, 5], [2, 6], [3, 9], [0, 0]], np.int32)
        ek, ev = k.copy(), v.copy()
        ek[5], ev[5] = k[1], v[1]
        ek[6], ev[6] = k[2], v[2]
        assert orc.copy_blocks(k, v, pairs) == 1
        assert k.tobytes() == ek.tobytes() and v.tobytes() == ev.tobytes()


def pin_swap_blocks(orc):
    """Swap between pools of different sizes: each destination block equals
    numpy's whole-block assignment from its source, every other block keeps
    its bytes, and a pair with an id outside its own pool is skipped."""
    rng = np.random.default_rng(12)
    B, Hkv, D = 4, 2, 8
    for dtype in ("f16", "bf16"):
        dk = to_storage(rng.standard_normal((9, B, Hkv, D)), dtype)
        dv = to_storage(rng.standard_normal((9, B, Hkv, D)), dtype)
        hk = poison((5, B, Hkv, D), dtype)
        hv = poison((5, B, Hkv, D), dtype)
        # device -> host: 7 is valid on the device, 4 on the host; 8 -> 5 and
        # 2 -> 6 name host blocks that do not exist, 9 a device block that does not
        pairs = np.array([[7, 4], [2, 0], [8, 5], [9, 1], [2, 6]], np.int32)
        ek, ev = hk.copy(), hv.copy()
        ek[4], ev[4] = dk[7], dv[7]
        ek[0], ev[0] = dk[2], dv[2]
        dk0, dv0 = dk.copy(), dv.copy()
        assert orc.swap_blocks(dk, dv, hk, hv, pairs) == 3
        assert hk.tobytes() == ek.tobytes() and hv.tobytes() == ev.tobytes()
        assert dk.tobytes() == dk0.tobytes() and dv.tobytes() == dv0.tobytes()
        # host -> device into other blocks
        back = np.array([[4, 1], [0, 8]], np.int32)
        ek, ev = dk.copy(), dv.copy()
        ek[1], ev[1] = dk0[7], dv0[7]
        ek[8], ev[8] = dk0[2], dv0[2]
        assert orc.swap_blocks(hk, hv, dk, dv, back) == 0
        assert dk.tobytes() == ek.tobytes() and dv.tobytes() == ev.tobytes()


def pin_swap_preserves_decode(orc):
    """"Paged Attention and the Block Manager", section "Running out of memory
    becomes a scheduling decision": a preempted sequence's blocks go out to
    host memory and come back later, into whichever blocks are free then. With
    its block table rewritten to the new blocks it decodes exactly as before,
    and as the contiguous attention over its tokens."""
    case = paged_case(13, [37, 50, 9], 8, 4, 2, 16, "bf16", spare_blocks=10)
    before = run_decode(orc, case)
    assert np.abs(before - brute_force(case)).max() < 1e-12
    s = 1
    n = -(-int(case["lens"][s]) // case["B"])
    victim = case["bt"][s, :n].copy()
    shape = (n + 2,) + case["k"].shape[1:]
    hk, hv = poison(shape, "bf16"), poison(shape, "bf16")
    host_ids = np.arange(2, n + 2, dtype=np.int32)
    assert orc.swap_blocks(case["k"], case["v"], hk, hv, np.stack([victim, host_ids], 1)) == 0
    used = set(case["bt"][case["bt"] >= 0].tolist())
    free = [b for b in range(case["NB"]) if b not in used]
    for b in victim:                       # the freed blocks are reused by others
        case["k"][b] = NAN_BITS_BF16
        case["v"][b] = NAN_BITS_BF16
    new_ids = np.array(free[:n], np.int32)
    assert orc.swap_blocks(hk, hv, case["k"], case["v"], np.stack([host_ids, new_ids], 1)) == 0
    case["bt"][s, :n] = new_ids
    after = run_decode(orc, case)
    assert after.tobytes() == before.tobytes()


def causal_brute_force(case, Q):
    """Contiguous causal attention with numpy/scipy: query row t of sequence s
    (its token at position t) attends over keys 0..t. Q[s]: [L_s][Hq][D] fp64."""
    g = case["Hq"] // case["Hkv"]
    outs = []
    for s, L in enumerate(case["lens"]):
        o = np.zeros((L, case["Hq"], case["D"]))
        for t in range(L):
            for h in range(case["Hq"]):
                K = case["Kc"][s][:t + 1, h // g]
                V = case["Vc"][s][:t + 1, h // g]
                o[t, h] = scipy.special.softmax(case["scale"] * (K @ Q[s][t, h])) @ V
        outs.append(o)
    return outs


def pin_prefill_chunks(orc):
    """"How a serving engine actually works", section "Prefill and decode are two
    different jobs": a prompt prefilled in chunks, one chunk per call, several
    sequences per call (some with no chunk in a round), gives every token the
    contiguous causal attention over the prompt up to and including itself."""
    chunking = [[5, 17, 1], [9], [1, 1, 30, 8], [16, 16]]
    lens = [sum(c) for c in chunking]
    for dtype, B, Hq, Hkv, D in (("f32", 8, 4, 2, 16), ("bf16", 4, 6, 2, 8), ("f16", 16, 2, 2, 8)):
        case = paged_case(31, lens, B, Hq, Hkv, D, dtype)
        rng = np.random.default_rng(32)
        Qs = [to_storage(rng.standard_normal((L, Hq, D)), dtype) for L in lens]
        want = causal_brute_force(case, [widen_lib(x, dtype) for x in Qs])
        done = [0] * len(lens)
        for r in range(max(len(c) for c in chunking)):
            sizes = [c[r] if r < len(c) else 0 for c in chunking]
            qs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
            ctx = np.array([done[s] + sizes[s] for s in range(len(lens))], np.int32)
            q = np.concatenate([Qs[s][done[s]:done[s] + sizes[s]] for s in range(len(lens))])
            got = orc.prefill(q, case["k"], case["v"], case["bt"], qs, ctx, case["scale"], dtype)
            for s in range(len(lens)):
                rows = got[qs[s]:qs[s + 1]]
                assert np.abs(rows - want[s][done[s]:ctx[s]]).max(initial=0) < 1e-12, (dtype, r, s)
                done[s] = int(ctx[s])
        assert done == lens


def pin_prefill_special_cases(orc):
    """A one-row chunk is decode at that length; the very first token of a
    prompt attends to itself alone, so its output is its own V row exactly;
    a chunk longer than its context is refused."""
    case = paged_case(33, [12, 7], 4, 4, 2, 8, "f32")
    rng = np.random.default_rng(34)
    q1 = to_storage(rng.standard_normal((2, 4, 8)), "f32")
    one = orc.prefill(q1, case["k"], case["v"], case["bt"], np.array([0, 1, 2], np.int32),
                      case["lens"], case["scale"], "f32")
    dec = orc.decode(q1, case["k"], case["v"], case["bt"], case["lens"], case["scale"], "f32")
    assert np.abs(one - dec).max() < 1e-12
    first = orc.prefill(q1, case["k"], case["v"], case["bt"], np.array([0, 1, 2], np.int32),
                        np.array([1, 1], np.int32), case["scale"], "f32")
    for s in range(2):
        for h in range(4):
            assert (first[s, h] == case["Vc"][s][0, h // 2]).all()
    try:
        orc.prefill(q1, case["k"], case["v"], case["bt"], np.array([0, 2, 2], np.int32),
                    np.array([1, 5], np.int32), case["scale"], "f32")
    except ValueError:
        pass
    else:
        raise AssertionError("a chunk longer than its context was accepted")


def pin_fork_copy_on_write(orc):
    """The serving page's fork: samples share the prompt's blocks; each sample's
    first token triggers a copy of the shared last block into a fresh one. After
    the copy and the append, every sample decodes like the contiguous
    attention over its own logical sequence."""
    from workloads.serving import BlockAllocator, Sequence
    rng = np.random.default_rng(9)
    B, Hkv, D, dtype = 16, 1, 8, "f32"
    alloc = BlockAllocator(16, B)
    prompt = Sequence("p", alloc)
    prompt.append_tokens(90)
    samples = [prompt.fork(f"s{i}") for i in range(4)]
    kpool = poison((16, B, Hkv, D), dtype)
    vpool = poison((16, B, Hkv, D), dtype)
    Kp = to_storage(rng.standard_normal((90, Hkv, D)), dtype)
    Vp = to_storage(rng.standard_normal((90, Hkv, D)), dtype)
    bt = np.array([prompt.table], np.int32)
    sm = orc.slot_mapping(bt, np.zeros(90, np.int32), np.arange(90, dtype=np.int32), B)
    orc.append(Kp, Vp, sm, kpool, vpool)
    q = to_storage(rng.standard_normal((4, 1, D)), dtype)
    tables, Ks, Vs = [], [], []
    for s in samples:
        shared_last = s.table[-1]
        s.append_tokens(1)
        assert s.table[-1] != shared_last
        orc.copy_blocks(kpool, vpool, [[shared_last, s.table[-1]]])
        kt = to_storage(rng.standard_normal((1, Hkv, D)), dtype)
        vt = to_storage(rng.standard_normal((1, Hkv, D)), dtype)
        tb = np.array([s.table], np.int32)
        orc.append(kt, vt, orc.slot_mapping(tb, [0], [90], B), kpool, vpool)
        tables.append(s.table)
        Ks.append(np.concatenate([widen_lib(Kp, dtype), widen_lib(kt, dtype)]))
        Vs.append(np.concatenate([widen_lib(Vp, dtype), widen_lib(vt, dtype)]))
    bts = np.array(tables, np.int32)
    lens = np.full(4, 91, np.int32)
    got = orc.decode(q, kpool, vpool, bts, lens, 1.0 / math.sqrt(D), dtype)
    ref = brute_force(dict(q=q, qc=widen_lib(q, dtype), Kc=Ks, Vc=Vs, Hkv=Hkv, lens=lens,
                           scale=1.0 / math.sqrt(D)))
    assert np.abs(got - ref).max() < 1e-12
    # the prompt's own blocks are untouched: it still decodes its 90 tokens
    got_p = orc.decode(q[:1], kpool, vpool, bt, np.array([90], np.int32), 1.0 / math.sqrt(D), dtype)
    ref_p = brute_force(dict(q=q[:1], qc=widen_lib(q[:1], dtype), Kc=[widen_lib(Kp, dtype)],
                             Vc=[widen_lib(Vp, dtype)], Hkv=Hkv, lens=np.array([90]),
                             scale=1.0 / math.sqrt(D)))
    assert np.abs(got_p - ref_p).max() < 1e-12


def pin_gather_order(orc):
    """Tokens appended through the slot mapping come back from the gather in
    logical order (row i of the gather holds the value written for position i)."""
    B, Hkv, D = 4, 2, 8
    case = paged_case(3, [1, 4, 5, 14], B, 2, Hkv, D, "f32")
    kpool = poison((case["NB"], B, Hkv, D), "f32")
    vpool = poison((case["NB"], B, Hkv, D), "f32")
    for s, L in enumerate(case["lens"]):
        pos = np.arange(L, dtype=np.int32)
        seq = np.full(L, s, np.int32)
        sm = orc.slot_mapping(case["bt"], seq, pos, B)
        rows = np.zeros((L, Hkv, D), np.float32)
        rows[:, :, 0] = pos[:, None] + 1000 * s
        rows[:, :, 1] = np.arange(Hkv)[None, :]
        orc.append(rows, rows, sm, kpool, vpool)
    for s, L in enumerate(case["lens"]):
        for h in range(Hkv):
            G = orc.gather(kpool, case["bt"], s, L, h, "f32")
            assert G[:, 0].tolist() == [i + 1000 * s for i in range(L)]
            assert (G[:, 1] == h).all()


# ---------------------------------------------------------------------------
# Decode attention.
# ---------------------------------------------------------------------------

def pin_decode_bruteforce(orc):
    """Equal to contiguous numpy/scipy attention on tiny inputs, all element types."""
    shapes = [([1, 3, 4, 5, 17], 4, 1, 1, 8),
              ([2, 7, 8, 9, 33], 8, 4, 2, 16),
              ([16, 1, 25], 16, 8, 1, 8),
              ([5, 12], 4, 6, 3, 4)]
    for i, (lens, B, Hq, Hkv, D) in enumerate(shapes):
        for dtype in ("f32", "f16", "bf16"):
            case = paged_case(100 + i, lens, B, Hq, Hkv, D, dtype)
            got = run_decode(orc, case)
            ref = brute_force(case)
            err = np.abs(got - ref).max()
            assert err < 1e-12, (lens, B, Hq, Hkv, D, dtype, err)


def pin_block_permutation_invariance(orc):
    """Renumbering physical blocks (data moved with them) changes nothing."""
    case = paged_case(21, [3, 17, 40, 9], 8, 4, 2, 16, "bf16")
    base = run_decode(orc, case)
    rng = np.random.default_rng(4)
    perm = rng.permutation(case["NB"])
    k2 = np.empty_like(case["k"])
    v2 = np.empty_like(case["v"])
    k2[perm] = case["k"]
    v2[perm] = case["v"]
    bt2 = np.where(case["bt"] >= 0, perm[np.maximum(case["bt"], 0)], -1).astype(np.int32)
    moved = dict(case, k=k2, v=v2, bt=bt2)
    assert np.array_equal(run_decode(orc, moved), base)


def pin_shared_prefix(orc):
    """Sequences that share prefix blocks (refcount > 1) give the same result
    as the same sequences holding private copies of those blocks."""
    B, Hkv, D, dtype = 4, 2, 8, "f16"
    case = paged_case(31, [13, 13, 13], B, 4, Hkv, D, dtype, spare_blocks=8)
    k, v, bt = case["k"].copy(), case["v"].copy(), case["bt"].copy()
    # make seqs 1 and 2 start with seq 0's first two blocks (8 tokens) as private copies
    spare = sorted(set(range(case["NB"])) - set(bt[bt >= 0].tolist()))
    for s in (1, 2):
        for j in range(2):
            k[bt[s, j]] = k[bt[0, j]]
            v[bt[s, j]] = v[bt[0, j]]
    private = dict(case, k=k, v=v, bt=bt)
    shared_bt = bt.copy()
    shared_bt[1:, :2] = bt[0, :2]
    shared = dict(case, k=k, v=v, bt=shared_bt)
    refs = np.bincount(shared_bt[shared_bt >= 0].ravel(), minlength=case["NB"])
    assert refs[bt[0, 0]] == 3 and spare
    assert np.array_equal(run_decode(orc, private), run_decode(orc, shared))


def pin_special_cases(orc):
    # one token: softmax weight 1, the output is that token's value exactly
    case = paged_case(41, [1, 1], 4, 2, 1, 8, "bf16")
    got = run_decode(orc, case)
    for s in range(2):
        for h in range(2):
            assert np.array_equal(got[s, h], case["Vc"][s][0, 0])
    # identical keys: uniform weights, the output is the mean of the values
    case = paged_case(42, [11], 4, 1, 1, 8, "f32")
    K = case["k"].copy()
    ids = case["bt"][0][case["bt"][0] >= 0]
    K[ids] = K[ids[0], 0]
    got = run_decode(orc, dict(case, k=K))
    assert np.abs(got[0, 0] - case["Vc"][0][:, 0].mean(axis=0)).max() < 1e-14
    # empty context: zeros, no NaN
    case = paged_case(43, [0, 5], 4, 2, 2, 8, "f32")
    got = run_decode(orc, case)
    assert (got[0] == 0).all() and np.isfinite(got[1]).all()
    # a query of zeros: uniform weights again
    case = paged_case(44, [7], 4, 1, 1, 8, "f32")
    q0 = np.zeros_like(case["q"])
    got = run_decode(orc, dict(case, q=q0))
    assert np.abs(got[0, 0] - case["Vc"][0][:, 0].mean(axis=0)).max() < 1e-14


def pin_partition_merge(orc):
    """Splitting the context and merging partition states is an identity."""
    case = paged_case(51, [45, 9], 4, 4, 2, 8, "f16")
    full = run_decode(orc, case)
    args = (case["q"], case["k"], case["v"], case["bt"], case["scale"], case["dtype"])
    for s, L in enumerate(case["lens"]):
        for qh in range(case["Hq"]):
            for P in (4, 8, 12, 64):
                cuts = list(range(0, L, P)) + [L]
                parts = [orc.decode_partition(*args, s, qh, a, b) for a, b in zip(cuts, cuts[1:])]
                o = np.array([p[0] for p in parts])
                m = np.array([p[1] for p in parts])
                l = np.array([p[2] for p in parts])
                merged = orc.lse_merge(m, l, o)
                assert np.abs(merged - full[s, qh]).max() < 1e-12, (s, qh, P)
            o1, m1, l1 = orc.decode_partition(*args, s, qh, 0, L)
            assert np.abs(o1 / l1 - full[s, qh]).max() < 1e-12
            oe, me, le = orc.decode_partition(*args, s, qh, 3, 3)
            assert me == -math.inf and le == 0 and (oe == 0).all()
            mixed = orc.lse_merge(np.array([me, m1]), np.array([le, l1]), np.stack([oe, o1]))
            assert np.abs(mixed - full[s, qh]).max() < 1e-12


ALL_PINS = [pin_f16_decoding, pin_bf16_decoding, pin_block_table_example, pin_slot_bijection,
            pin_append_scatter, pin_copy_blocks, pin_swap_blocks, pin_swap_preserves_decode,
            pin_fork_copy_on_write, pin_gather_order, pin_prefill_chunks, pin_prefill_special_cases,
            pin_decode_bruteforce,
            pin_block_permutation_invariance, pin_shared_prefix, pin_special_cases,
            pin_partition_merge]
