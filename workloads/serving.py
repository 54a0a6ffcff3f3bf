"""Host-side block manager and continuous-batching scheduler that generate the
continuous-batching workload (which physical blocks each sequence holds,
which tokens each step appends, which sequences each step decodes).

Behaviour follows the pages; the code is this package's own:

* BlockAllocator: a FIFO free list of physical block ids plus reference
  counts ("How a serving engine actually works", section "The code"; "Paged
  Attention and the Block Manager", section "The build": n_blocks and
  block_size must be positive). allocate() takes the head of the free list and
  raises OutOfBlocks when it is empty; share() bumps a count ("Paged-KV +
  Continuous Batching From Scratch", section 1); free_block() returns a block
  to the tail of the free list only when its last reference goes (the
  reference-counting guard) and refuses a double free (section 2 of the same
  page); copy_on_write() keeps a block its sole owner writes into and
  otherwise hands out a fresh one (the data copy itself is the device's job).
* Sequence: a block table plus a token count; growing by one token takes a
  new block exactly when the token starts one, otherwise writes into the last
  block (copy-on-write if shared); fork() shares every block; release() drops
  every reference.
* ContinuousBatcher: each step admits waiting requests that have arrived, in
  order, while slots remain and their blocks fit, counting blocks already
  promised this step (ch08 page, "The build": the `reserved` counter, and stop
  at the first request that does not fit); grows every running sequence by one
  token; when the pool is empty, preempts the most recently admitted sequence
  (Tessera page section 3: LIFO), releases all its blocks and puts it at the
  front of the waiting queue with its tokens intact, to be recomputed (its
  KV re-appended) on re-admission ("Paged Attention and the Block Manager",
  section "Running out of memory becomes a scheduling decision"). With
  preempt="swap" (the other choice that section names) the victim's blocks
  are copied out to a host pool instead and copied back into free device
  blocks on re-admission, so nothing is re-appended; a victim whose KV was
  not written yet (admitted by recompute in the same step) or that does not
  fit in the host pool is recomputed.

Nothing here computes a slot or touches K/V values: a step plan lists
(request, position) pairs and block tables; the slot mapping, append and
decode run on whichever side consumes the plan.
"""
from collections import deque
from dataclasses import dataclass, field

import numpy as np


class OutOfBlocks(RuntimeError):
    pass


class DoubleFree(RuntimeError):
    pass


class BlockAllocator:
    def __init__(self, n_blocks, block_size):
        if n_blocks < 1 or block_size < 1:
            raise ValueError(f"a pool needs at least one block of at least one token "
                             f"(got {n_blocks} blocks of {block_size})")
        self.n_blocks = int(n_blocks)
        self.block_size = int(block_size)
        self._free = deque(range(self.n_blocks))
        self._ref = [0] * self.n_blocks
        self.cow_copies = 0

    @property
    def n_free(self):
        return len(self._free)

    def free_list(self):
        return list(self._free)

    def refcount(self, b):
        return self._ref[b]

    def blocks_needed(self, n_tokens):
        return -(-int(n_tokens) // self.block_size)

    def allocate(self):
        if not self._free:
            raise OutOfBlocks("no free physical blocks")
        b = self._free.popleft()
        self._ref[b] = 1
        return b

    def share(self, b):
        if self._ref[b] < 1:
            raise ValueError(f"block {b} is not allocated")
        self._ref[b] += 1
        return b

    def free_block(self, b):
        """Drop one reference; True when the block went back to the pool."""
        if self._ref[b] < 1:
            raise DoubleFree(f"block {b} freed with no reference left")
        self._ref[b] -= 1
        if self._ref[b] == 0:
            self._free.append(b)
            return True
        return False

    def copy_on_write(self, b):
        """(block to write into, whether a fresh block replaced a shared one)."""
        if self._ref[b] == 1:
            return b, False
        fresh = self.allocate()
        self._ref[b] -= 1
        self.cow_copies += 1
        return fresh, True


class Sequence:
    def __init__(self, name, alloc):
        self.name = name
        self.alloc = alloc
        self.table = []
        self.n_tokens = 0

    def append_tokens(self, n):
        """Grow by n tokens; returns the number of copy-on-write events."""
        cows = 0
        for _ in range(int(n)):
            if self.n_tokens % self.alloc.block_size == 0:
                self.table.append(self.alloc.allocate())
            else:
                self.table[-1], copied = self.alloc.copy_on_write(self.table[-1])
                cows += int(copied)
            self.n_tokens += 1
        return cows

    def fork(self, name):
        child = Sequence(name, self.alloc)
        child.table = [self.alloc.share(b) for b in self.table]
        child.n_tokens = self.n_tokens
        return child

    def release(self):
        for b in self.table:
            self.alloc.free_block(b)
        self.table = []

    def waste(self):
        return len(self.table) * self.alloc.block_size - self.n_tokens


# ---------------------------------------------------------------------------
# Continuous batching over a synthetic request stream
# ---------------------------------------------------------------------------

OUTPUT_LENGTHS = (8, 16, 32, 64, 128)
OUTPUT_WEIGHTS = (0.30, 0.25, 0.15, 0.15, 0.15)


@dataclass
class Request:
    rid: int
    arrival: int
    prompt_len: int
    output_len: int
    generated: int = 0
    admitted_at: list = field(default_factory=list)
    finished_at: int = -1
    preemptions: int = 0
    delivered: list = field(default_factory=list)   # positions whose token was handed out

    @property
    def n_tokens(self):
        return self.prompt_len + self.generated

    @property
    def done(self):
        return self.generated >= self.output_len


def synthetic_requests(n=64, seed=11, prompt_lo=32, prompt_hi=512, rate=1.0):
    """Poisson arrivals (mean `rate` per step), prompts uniform in
    [prompt_lo, prompt_hi], outputs drawn from OUTPUT_LENGTHS with OUTPUT_WEIGHTS."""
    rng = np.random.default_rng(seed)
    gaps = rng.exponential(1.0 / rate, size=n)
    arrivals = np.floor(np.cumsum(gaps) - gaps[0]).astype(int)
    prompts = rng.integers(prompt_lo, prompt_hi, size=n, endpoint=True)
    outputs = rng.choice(OUTPUT_LENGTHS, size=n, p=OUTPUT_WEIGHTS)
    return [Request(i, int(a), int(p), int(o)) for i, (a, p, o) in
            enumerate(zip(arrivals, prompts, outputs))]


@dataclass
class StepPlan:
    """One decode step of the running set.

    rids[b]         request decoded in batch row b (admission order)
    block_tables    int32 [R][max_blocks], -1 past each sequence's blocks
    context_lens    int32 [R]: tokens attended over (the step's token included)
    token_row,
    token_pos       int32 [T]: tokens whose K/V this step appends (batch row, position):
                    the whole history of sequences (re)admitted this step by
                    recompute, then one new token per running sequence
    query_pos       int32 [R]: position of each row's query token
    swap_in         int32 [n][2]: (host block, device block) copied in this step
    swap_out        int32 [n][2]: (device block, host block) copied out this step

    On the device a step runs swap_in, then swap_out, then the append, then the
    decode: a sequence swapped in and preempted again in one step is copied
    back out after it arrived, a host block freed by a swap-in is read before a
    swap-out reuses it, and a device block freed by a swap-out is read before
    an append reuses it.
    """
    step: int
    rids: list
    block_tables: np.ndarray
    context_lens: np.ndarray
    token_row: np.ndarray
    token_pos: np.ndarray
    query_pos: np.ndarray
    admitted: list
    preempted: list
    swap_in: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), np.int32))
    swap_out: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), np.int32))


class ContinuousBatcher:
    def __init__(self, requests, slots, n_blocks, block_size, max_blocks=None,
                 preempt="recompute", host_blocks=0):
        if preempt not in ("recompute", "swap"):
            raise ValueError("preempt must be 'recompute' or 'swap'")
        self.requests = {r.rid: r for r in requests}
        self.alloc = BlockAllocator(n_blocks, block_size)
        self.preempt = preempt
        self.host = BlockAllocator(host_blocks, block_size) if preempt == "swap" else None
        self.swapped = {}            # rid -> (host block table, tokens held)
        self.swapped_out_blocks = 0
        self.swapped_in_blocks = 0
        self._recomputed = set()     # admitted by recompute this step: KV not written yet
        self._swap_in, self._swap_out = [], []
        self.waiting = deque(sorted(requests, key=lambda r: (r.arrival, r.rid)))
        self.running = []            # admission order, oldest first
        self.seqs = {}
        self.slots = int(slots)
        self.step = 0
        longest = max(r.prompt_len + r.output_len for r in requests)
        self.max_blocks = max_blocks or self.alloc.blocks_needed(longest)
        self.total_preemptions = 0

    def idle(self):
        return not self.waiting and not self.running

    def _admit(self):
        admitted = []
        reserved = 0
        while (self.waiting and len(self.running) + len(admitted) < self.slots
               and self.waiting[0].arrival <= self.step):
            cand = self.waiting[0]
            need = self.alloc.blocks_needed(cand.n_tokens + 1)
            if need > self.alloc.n_free - reserved:
                break                      # leave it queued; do not skip ahead
            reserved += need
            admitted.append(self.waiting.popleft())
        for r in admitted:
            seq = Sequence(r.rid, self.alloc)
            held = self.swapped.pop(r.rid, None)
            if held is None:
                seq.append_tokens(r.n_tokens)  # recompute: the whole history is re-appended
                self._recomputed.add(r.rid)
            else:
                host_table, n_tokens = held    # swap in: same tokens, fresh device blocks
                for hb in host_table:
                    db = self.alloc.allocate()
                    seq.table.append(db)
                    self._swap_in.append((hb, db))
                    self.host.free_block(hb)
                seq.n_tokens = n_tokens
                self.swapped_in_blocks += len(host_table)
            self.seqs[r.rid] = seq
            r.admitted_at.append(self.step)
            self.running.append(r)
        return admitted

    def _preempt_one(self, protect):
        for r in reversed(self.running):   # newest admission first
            if r.rid != protect:
                self.running.remove(r)
                seq = self.seqs.pop(r.rid)
                # tokens on the device: a victim that already grew this step
                # has not had that token appended yet (appends follow swap-outs)
                written = r.n_tokens
                keep = self.alloc.blocks_needed(written)
                if (self.preempt == "swap" and r.rid not in self._recomputed
                        and self.host.n_free >= keep):
                    host_table = [self.host.allocate() for _ in range(keep)]
                    self._swap_out.extend(zip(seq.table[:keep], host_table))
                    self.swapped[r.rid] = (host_table, written)
                    self.swapped_out_blocks += keep
                seq.release()
                r.preemptions += 1
                self.total_preemptions += 1
                self.waiting.appendleft(r)
                return r
        raise OutOfBlocks("a single sequence does not fit in the pool")

    def schedule(self):
        """Plan the next step, or return None when every request is done."""
        self._recomputed = set()
        self._swap_in, self._swap_out = [], []
        admitted = self._admit()
        while not self.running:
            if not self.waiting:
                return None
            if self.waiting[0].arrival <= self.step:
                raise OutOfBlocks("a waiting request does not fit in the empty pool")
            self.step = self.waiting[0].arrival      # idle until the next arrival
            admitted = self._admit()
        admitted_ids = {r.rid for r in admitted}
        history = {r.rid: r.n_tokens for r in admitted if r.rid in self._recomputed}
        preempted = []
        # grow every running sequence by the token this step writes
        for r in list(self.running):
            if r not in self.running:
                continue
            seq = self.seqs[r.rid]
            while True:
                try:
                    seq.append_tokens(1)
                    break
                except OutOfBlocks:
                    preempted.append(self._preempt_one(protect=r.rid).rid)
        rows = {r.rid: b for b, r in enumerate(self.running)}
        R = len(self.running)
        bt = np.full((R, self.max_blocks), -1, dtype=np.int32)
        lens = np.zeros(R, dtype=np.int32)
        qpos = np.zeros(R, dtype=np.int32)
        tok_row, tok_pos = [], []
        for b, r in enumerate(self.running):
            seq = self.seqs[r.rid]
            bt[b, :len(seq.table)] = seq.table
            lens[b] = seq.n_tokens
            qpos[b] = seq.n_tokens - 1
            if r.rid in admitted_ids and r.rid in history:
                tok_row.extend([b] * history[r.rid])
                tok_pos.extend(range(history[r.rid]))
        for b, r in enumerate(self.running):
            tok_row.append(b)
            tok_pos.append(self.seqs[r.rid].n_tokens - 1)
        plan = StepPlan(self.step, [r.rid for r in self.running], bt, lens,
                        np.asarray(tok_row, np.int32), np.asarray(tok_pos, np.int32), qpos,
                        [rid for rid in admitted_ids if rid in rows], preempted,
                        np.asarray(self._swap_in, np.int32).reshape(-1, 2),
                        np.asarray(self._swap_out, np.int32).reshape(-1, 2))
        return plan

    def commit(self, plan):
        """Finish the step: every decoded sequence hands out one token."""
        for rid in plan.rids:
            r = self.requests[rid]
            r.delivered.append(r.n_tokens)     # the position of the token handed out
            r.generated += 1
        for r in [r for r in self.running if r.done]:
            self.running.remove(r)
            self.seqs.pop(r.rid).release()
            r.finished_at = self.step
        self.step += 1

    def run(self):
        """All step plans of the trace (host bookkeeping only)."""
        plans = []
        while True:
            plan = self.schedule()
            if plan is None:
                return plans
            plans.append(plan)
            self.commit(plan)
