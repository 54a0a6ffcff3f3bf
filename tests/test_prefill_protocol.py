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


def make_items(cta, grid, before, chunk, g, n_kv, parts=1, min_part=MIN_PART_TILES):
    """The items of CTA `cta`, in the kernel's order (key parts innermost; an
    item's keys in at most ceil(N / min_part) parts)."""
    lens = [b + c for b, c in zip(before, chunk)]
    qs = np.concatenate([[0], np.cumsum(chunk)])
    tq = ROWS // g                  # whole tokens per Q tile
    tile_tokens = 2 * tq
    tiles = -(-max(chunk) // tile_tokens)
    S = len(chunk)
    ranked = sorted(range(S), key=lambda s: (-lens[s], s)) if S > 1 else list(range(S))
    per_tile = n_kv * parts
    per_seq = tiles * per_tile
    num_items = S * per_seq
    items, m = [], 0
    while True:
        k = m * grid + ((grid - 1 - cta) if (m & 1) else cta)
        m += 1
        if k >= num_items:
            return items
        r, rem = divmod(k, per_seq)
        s = ranked[r]
        qt = tiles - 1 - rem // per_tile
        part = rem % per_tile % parts
        n, L = int(qs[s + 1] - qs[s]), lens[s]
        j0 = qt * tile_tokens
        if j0 >= n:
            continue
        ntok = min(tile_tokens, n - j0)
        pos0 = L - n + j0
        nk = [(pos0 + t * tq + min(ntok - t * tq, tq) - 1) // KEYS + 1 if ntok > t * tq else 0
              for t in range(TILES)]
        N = nk[1] if nk[1] > 0 else nk[0]
        eff = min(parts, max(1, -(-N // min_part)))
        if part >= eff:
            continue
        kb, ke = N * part // eff, N * (part + 1) // eff
        items.append(dict(nk=[max(min(x, ke) - kb, 0) for x in nk], nkt=ke - kb,
                          tail=ke == N and N * KEYS > L))


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
@pytest.mark.parametrize("grid,parts", [(1, 1), (5, 1), (37, 1), (5, 3), (37, 3)])
def test_no_deadlock_or_phase_hazard(g, n_kv, grid, parts):
    """Chunks of one row to three query tiles, contexts on a 64-key boundary
    and ragged, second Q tiles empty: every interleaving tried ends, with no
    barrier two phases past a waiter or one behind it (groups that divide 128
    and 3, whose Q tiles hold 42 whole tokens), whole items and items whose
    keys are split in up to three parts (a part's first tile past a tile's
    rows, a tail only in the last part; parts of one key tile or more, to split
    far more items than the kernel's rule of one part per 16 key tiles would)."""
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
