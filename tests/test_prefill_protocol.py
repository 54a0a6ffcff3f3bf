"""The persistent tcgen05 prefill kernel's barrier protocol, modelled on the CPU.

Each role of a CTA (producer, Q-copy/V-zeroing warp, the two MMA issuers, the
two tiles' softmax warps) is a generator that performs its arrivals and yields
its mbarrier waits in the kernel's order, with the phase index each wait means;
copies and MMAs complete at once. A scheduler runs the roles in random order.
The test fails if the CTA stops with roles still waiting (a deadlock), or if a
barrier is ever two or more phases past one of its waiters, or a phase behind
it (a parity wait could then never pass, or pass early). The items come from
the kernel's own ordering rules (sequences ranked by context length, bands
dealt in alternating directions, query tiles from the last, then kv heads).

A model, not the kernel: when the kernel's waits or arrivals change, this
model must change with them. One case puts back an earlier protocol (an "O
free" barrier the issuer waited on, with Q copied by TMA) and checks that the
model finds its phase hazard.
"""
import numpy as np
import pytest

KEYS, ROWS, TILES, STAGES = 64, 128, 2, 4
MIN_PART_TILES = 16   # the kernel's least key tiles per part of a split item


class Hazard(Exception):
    pass


class Barrier:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.tx = 0
        self.phase = 0          # completed phases

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, "more arrivals than the barrier's count"
        self._complete()

    def expect(self, n):
        self.tx += n

    def land(self, n):
        self.tx -= n
        self._complete()

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def passes(self, n):
        """A parity wait for phase n (negative: a phase before the first). It
        is only sound while phase n - 1 has completed and phase n + 1 has not."""
        if self.phase >= n + 2:
            raise Hazard("barrier two phases past its waiter")
        if self.phase < n:
            raise Hazard("barrier one phase behind its waiter: the wait would pass early")
        return (self.phase & 1) != (n & 1)


def item_tiles(before, chunk, g, n_kv):
    """Every item in the shared order without ranking (sequence, query tile
    from the last, kv head): (L, pos0, ntok, nk per Q tile, N key tiles)."""
    lens = [b + c for b, c in zip(before, chunk)]
    tq = ROWS // g                  # whole tokens per Q tile
    tile_tokens = 2 * tq
    tiles = -(-max(chunk) // tile_tokens)
    out = []
    for s in range(len(chunk)):
        for qt in range(tiles - 1, -1, -1):
            for _ in range(n_kv):
                n, L = chunk[s], lens[s]
                j0 = qt * tile_tokens
                if j0 >= n:
                    out.append(None)
                    continue
                ntok = min(tile_tokens, n - j0)
                pos0 = L - n + j0
                nk = [(pos0 + t * tq + min(ntok - t * tq, tq) - 1) // KEYS + 1 if ntok > t * tq else 0
                      for t in range(TILES)]
                out.append((L, pos0, ntok, nk, nk[1] if nk[1] > 0 else nk[0]))
    return out


PIECE_COST = 4   # the plan's fixed cost of a piece, in key tiles
MAX_ITEM_PARTS = 16  # parts per item in the parts layout at most


def split_plan(Ns, grid, parts, min_part=MIN_PART_TILES):
    """The key split's plan: (r, pp, off, T); pp > 0 picks the parts layout
    (pp CTAs per item), else ranges of r tiles of all items end to end."""
    off = np.concatenate([[0], np.cumsum(Ns)]).astype(int)
    T, mx = int(off[-1]), max(Ns, default=0)
    r = -(-T // grid)
    if mx > 1:
        r = max(r, (mx - 2) // (parts - 1) + 1)
    r = max(r, max(min(min_part, mx), 1))
    pp = min(parts, MAX_ITEM_PARTS, grid // max(len(Ns), 1))
    if pp > 0:
        part_mx = max((-(-n // part_count(n, pp, min_part)) for n in Ns), default=0)
        if part_mx + PIECE_COST > r + 2 * PIECE_COST:
            pp = 0
    return r, pp, off, T


def part_count(n, pp, min_part=MIN_PART_TILES):
    return min(pp, max(1, -(-n // min_part)))


def split_pieces(cta, plan, Ns, min_part=MIN_PART_TILES):
    """The pieces of CTA `cta`, in order: (item, kb, ke, slot, split)."""
    r, pp, off, T = plan
    if pp > 0:
        i, q = divmod(cta, pp)
        if i >= len(Ns) or Ns[i] == 0 or q >= part_count(Ns[i], pp, min_part):
            return []
        e = part_count(Ns[i], pp, min_part)
        start, end = off[i] + Ns[i] * q // e, off[i] + Ns[i] * (q + 1) // e
    else:
        start = min(cta * r, T)
        end = min(start + r, T)
    out = []
    for i, N in enumerate(Ns):
        kb, ke = max(start - off[i], 0), min(end - off[i], N)
        if ke > kb:
            out.append((i, kb, ke, 2 * cta + (0 if kb > 0 else 1), kb > 0 or ke < N))
    return out


def merge_word(i, plan, Ns, min_part=MIN_PART_TILES):
    """The merge's (first CTA, piece count) of item i."""
    r, pp, off, T = plan
    N = Ns[i]
    if N == 0:
        return 0, 0
    if pp > 0:
        return i * pp, part_count(N, pp, min_part)
    c0 = off[i] // r
    return c0, (off[i] + N - 1) // r - c0 + 1


def make_items(cta, grid, before, chunk, g, n_kv, parts=1, min_part=MIN_PART_TILES):
    """The items of CTA `cta`, in the kernel's order. Whole items (parts 1):
    sequences ranked by length, bands dealt in alternating directions. Key
    split: the pieces of the CTA's range of the call's key tiles."""
    if parts > 1:
        its = item_tiles(before, chunk, g, n_kv)
        Ns = [0 if x is None else x[4] for x in its]
        plan = split_plan(Ns, grid, parts, min_part)
        items = []
        for i, kb, ke, _, _ in split_pieces(cta, plan, Ns, min_part):
            L, _, _, nk, N = its[i]
            items.append(dict(nk=[max(min(x, ke) - kb, 0) for x in nk], nkt=ke - kb,
                              tail=ke == N and N * KEYS > L))
        return items
    lens = [b + c for b, c in zip(before, chunk)]
    qs = np.concatenate([[0], np.cumsum(chunk)])
    tq = ROWS // g                  # whole tokens per Q tile
    tile_tokens = 2 * tq
    tiles = -(-max(chunk) // tile_tokens)
    S = len(chunk)
    ranked = sorted(range(S), key=lambda s: (-lens[s], s)) if S > 1 else list(range(S))
    per_seq = tiles * n_kv
    num_items = S * per_seq
    items, m = [], 0
    while True:
        k = m * grid + ((grid - 1 - cta) if (m & 1) else cta)
        m += 1
        if k >= num_items:
            return items
        r, rem = divmod(k, per_seq)
        s = ranked[r]
        qt = tiles - 1 - rem // n_kv
        n, L = int(qs[s + 1] - qs[s]), lens[s]
        j0 = qt * tile_tokens
        if j0 >= n:
            continue
        ntok = min(tile_tokens, n - j0)
        pos0 = L - n + j0
        nk = [(pos0 + t * tq + min(ntok - t * tq, tq) - 1) // KEYS + 1 if ntok > t * tq else 0
              for t in range(TILES)]
        N = nk[1] if nk[1] > 0 else nk[0]
        items.append(dict(nk=nk, nkt=N, tail=N * KEYS > L))


def run_cta(items, rng, ofree=False):
    """Runs one CTA's roles to the end; returns the roles left waiting (empty
    when every role finished)."""
    bars = {}

    def B(name, count=1):
        if name not in bars:
            bars[name] = Barrier(count)
        return bars[name]

    for st in range(STAGES):
        B(("full", st)), B(("empty", st), TILES), B(("tailv", st))

    def producer():
        kt = 0
        for it in items:
            for j in range(it["nkt"]):
                gk = kt + j
                st = gk % STAGES
                yield ("empty", st), gk // STAGES - 1
                if not (it["tail"] and j == it["nkt"] - 1):
                    B(("full", st)).expect(2)
                    B(("full", st)).arrive()
                    B(("full", st)).land(2)
                else:
                    # K on the stage's barrier (armed, no arrival); V on the tail barrier
                    B(("full", st)).expect(1)
                    B(("tailv", st)).expect(1)
                    B(("tailv", st)).arrive()
                    B(("full", st)).land(1)
                    B(("tailv", st)).land(1)
            kt += it["nkt"]

    def copy_and_zero():
        kt = 0
        tail_phase = [0] * STAGES
        for i, it in enumerate(items):
            for t in range(TILES):
                if i > 0:
                    yield ("qfree", t), i - 1
                if it["nk"][t] > 0:
                    B(("qfull", t)).expect(1)
                    B(("qfull", t)).arrive()
                    B(("qfull", t)).land(1)
                else:
                    B(("qfull", t)).arrive()
            if it["tail"]:
                st = (kt + it["nkt"] - 1) % STAGES
                yield ("tailv", st), tail_phase[st]
                tail_phase[st] += 1
                B(("full", st)).arrive()
            kt += it["nkt"]

    def issuer(t):
        kt = jt = 0
        for i, it in enumerate(items):
            nk = it["nk"][t]
            yield ("qfull", t), i
            if nk > 0:
                for j in range(min(2, nk)):
                    yield ("full", (kt + j) % STAGES), (kt + j) // STAGES
                    B(("s", t, (jt + j) & 1)).arrive()
                if nk <= 2:
                    B(("qfree", t)).arrive()
            for j in range(it["nkt"]):
                gk = kt + j
                if j < nk:
                    yield ("p", t, (jt + j) & 1), (jt + j) >> 1
                    if ofree and j == 0 and i > 0:
                        yield ("ofree", t), i - 1
                    # beside the P wait, a look (no wait) at the K/V of key tile j + 2
                    ahead = j + 2 < nk
                    full2 = ("full", (gk + 2) % STAGES), (gk + 2) // STAGES
                    kv_in = ahead and B(full2[0]).passes(full2[1])
                    B(("o", t, (jt + j) & 1)).arrive()
                    B(("empty", gk % STAGES)).arrive()
                    if ahead:
                        if not kv_in:
                            yield full2
                        B(("s", t, (jt + j + 2) & 1)).arrive()
                        if j + 2 == nk - 1:
                            B(("qfree", t)).arrive()
                else:
                    yield ("full", gk % STAGES), gk // STAGES
                    B(("empty", gk % STAGES)).arrive()
            if nk == 0:
                if ofree and i > 0:
                    yield ("ofree", t), i - 1
                B(("qfree", t)).arrive()
            kt += it["nkt"]
            jt += nk

    def softmax(t):
        jt = prev_nk = prev_end = 0
        for i, it in enumerate(items):
            nk = it["nk"][t]
            if i > 0:
                if prev_nk:
                    yield ("o", t, (prev_end - 1) & 1), (prev_end - 1) >> 1
                if ofree:
                    B(("ofree", t)).arrive()
            for j in range(nk):
                gj = jt + j
                yield ("s", t, gj & 1), gj >> 1
                B(("p", t, gj & 1)).arrive()
            prev_nk, prev_end = nk, jt + nk
            jt += nk
        if items and prev_nk:
            yield ("o", t, (prev_end - 1) & 1), (prev_end - 1) >> 1

    roles = {"producer": producer(), "copy_zero": copy_and_zero(), "issuer0": issuer(0),
             "issuer1": issuer(1), "softmax0": softmax(0), "softmax1": softmax(1)}
    waiting = dict.fromkeys(roles)
    while roles:
        for w in waiting.values():
            if w is not None:
                B(w[0]).passes(w[1])          # the hazard check, on every blocked wait
        ready = [r for r in roles if waiting[r] is None or B(waiting[r][0]).passes(waiting[r][1])]
        if not ready:
            return {r: waiting[r] for r in roles}
        r = ready[rng.integers(len(ready))]
        try:
            waiting[r] = next(roles[r])
        except StopIteration:
            del roles[r], waiting[r]
    return {}


def many_items_workload():
    rng = np.random.default_rng(520)
    before = rng.integers(0, 900, size=40)
    chunk = rng.integers(1, 600, size=40)
    before[:4] = [0, 64, 128, 0]
    chunk[:4] = [64, 64, 128, 100]
    return before.tolist(), chunk.tolist()


def check(before, chunk, g, n_kv, grid, seeds, ofree=False, parts=1, min_part=MIN_PART_TILES):
    for cta in range(grid):
        items = make_items(cta, grid, before, chunk, g, n_kv, parts, min_part)
        for seed in range(seeds):
            left = run_cta(items, np.random.default_rng(seed), ofree=ofree)
            assert not left, f"cta {cta} seed {seed}: deadlock, waiting {left}"


@pytest.mark.parametrize("g,n_kv", [(1, 8), (3, 4), (8, 4), (64, 1)])
@pytest.mark.parametrize("grid,parts", [(1, 1), (5, 1), (37, 1), (5, 3), (37, 3), (152, 32)])
def test_no_deadlock_or_phase_hazard(g, n_kv, grid, parts):
    """Chunks of one row to three query tiles, contexts on a 64-key boundary
    and ragged, second Q tiles empty: every interleaving tried ends, with no
    barrier two phases past a waiter or one behind it (groups that divide 128
    and 3, whose Q tiles hold 42 whole tokens), whole items and the key split's
    pieces (a piece's first tile past a tile's rows, a tail only in an item's
    last piece, a range holding the end of one item and the start of the next;
    ranges of one key tile or more, to cut far more items than the kernel's
    floor of 16 tiles would)."""
    before, chunk = many_items_workload()
    check(before, chunk, g, n_kv, grid, seeds=3, parts=parts, min_part=1 if parts > 1 else MIN_PART_TILES)


def test_model_finds_the_removed_o_free_hazard():
    """The protocol with an "O free" barrier (the softmax warps arrive once
    they have read an item's O; the issuer waits before the item's first P V,
    or at the end of an item it has no MMA in) and Q copied by TMA: a tile
    with no rows in several items lets the softmax warps run two phases ahead."""
    before, chunk = many_items_workload()
    with pytest.raises(Hazard):
        check(before, chunk, 1, 8, 37, seeds=3, ofree=True)


def kernel_and_merge_agree(Ns, grid, parts, min_part=MIN_PART_TILES):
    plan = split_plan(Ns, grid, parts, min_part)
    r, pp, off, T = plan
    if pp == 0:
        assert r * grid >= T
    seen = {}                      # item -> [(cta, kb, ke, slot, split)] from the kernel's side
    slots = set()
    for c in range(grid):
        ps = split_pieces(c, plan, Ns, min_part)
        if pp > 0:
            assert len(ps) <= 1
        else:
            # the CTA's first item and piece count as the kernel finds them (binary searches)
            start = min(c * r, T)
            end = min(start + r, T)
            first = next((i for i in range(len(Ns)) if off[i + 1] > start), len(Ns))
            last = next((i for i in range(first, len(Ns)) if off[i + 1] >= end), len(Ns))
            count = last - first + 1 if start < end else 0
            assert [i for i, *_ in ps] == [i for i in range(first, first + count) if Ns[i] > 0]
        for i, kb, ke, slot, split in ps:
            assert 0 <= slot < 2 * grid
            if split:
                assert slot not in slots, "two pieces in one slot"
                slots.add(slot)
            seen.setdefault(i, []).append((c, kb, ke, slot, split))
    for i, N in enumerate(Ns):
        got = seen.get(i, [])
        # every key tile of the item exactly once, in order
        assert sum(ke - kb for _, kb, ke, _, _ in got) == N
        assert all(a[2] == b[1] for a, b in zip(got, got[1:]))
        assert len(got) <= parts
        c0, n = merge_word(i, plan, Ns, min_part)
        assert n == len(got)
        if N == 0:
            continue
        assert [g_[0] for g_ in got] == list(range(c0, c0 + n))
        assert all(split == (n > 1) for *_, split in got)
        if n > 1:
            assert [slot for *_, slot, _ in got] == [2 * (c0 + q) + (1 if q == 0 else 0) for q in range(n)]
    return pp


@pytest.mark.parametrize("grid", [1, 7, 37, 152])
@pytest.mark.parametrize("parts", [2, 3, 32])
def test_key_split_plan(grid, parts):
    """The key split's pieces, as the kernel cuts them (ranges or parts,
    whichever the plan picks) and as the merge finds them: every key tile
    once, no item in more than `parts` pieces, each piece of a cut item in a
    slot of its own below 2 x grid, the merge's first CTA, piece count and
    slots those of the kernel's pieces; items of no tiles, one long item among
    short ones, and all-empty calls."""
    rng = np.random.default_rng(grid * 100 + parts)
    cases = [[258] * 32, [257] * 8, [34] * 32, [0] * 5, [1] * 40, [5000] + [3] * 60, [0, 16, 0, 17, 0],
             list(rng.integers(0, 600, 500)), list(rng.integers(0, 3, 200)), [2] * 32,
             [315] * 32 + [49] * 32, [130] * 128]
    layouts = [kernel_and_merge_agree([int(x) for x in Ns], grid, parts) > 0 for Ns in cases]
    if grid == 152 and parts == 32:
        # equal items that divide the SMs take parts; one long item among short ones ranges
        assert layouts[1] and layouts[2] and not layouts[0] and not layouts[5] and not layouts[10]


@pytest.mark.parametrize("g,n_kv", [(1, 4), (3, 2), (8, 2)])
def test_no_deadlock_in_the_parts_layout(g, n_kv):
    """Few equal items over long contexts (the plan takes parts: one piece per
    CTA, a part's first tile past the first Q tile's rows): every interleaving
    tried ends without a phase hazard."""
    before, chunk = [3000, 3000], [100, 37]
    its = item_tiles(before, chunk, g, n_kv)
    Ns = [0 if x is None else x[4] for x in its]
    assert split_plan(Ns, 152, 32)[1] > 0
    check(before, chunk, g, n_kv, 152, seeds=2, parts=32)
