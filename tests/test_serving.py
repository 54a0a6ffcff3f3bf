"""Host-side block manager and scheduler against the pages' printed examples
and the invariants the pages state (CPU only)."""
import pytest

from oracle_pins import read_golden
from workloads.serving import (BlockAllocator, ContinuousBatcher, DoubleFree, OutOfBlocks, Sequence,
                               synthetic_requests)

KIB_PER_TOKEN_LLAMA2_7B = 512      # "Reserving memory you will never write": 512 KiB per token


def test_allocator_validates_its_sizes():
    with pytest.raises(ValueError):
        BlockAllocator(0, 16)
    with pytest.raises(ValueError):
        BlockAllocator(8, 0)


def test_copy_on_write_fork_example():
    rows = {r[0]: r for r in read_golden("cow_fork.txt")}
    B = int(rows["block_size"][1])
    alloc = BlockAllocator(64, B)
    prompt = Sequence("prompt", alloc)
    prompt.append_tokens(int(rows["prompt_tokens"][1]))
    want_blocks = [int(x) for x in rows["prompt_tokens"][3:rows["prompt_tokens"].index("used")]]
    assert prompt.table == want_blocks
    used = lambda: sum(alloc.refcount(b) > 0 for b in range(alloc.n_blocks))
    assert used() == int(rows["prompt_tokens"][-1])
    fork = rows["fork"]
    samples = [prompt.fork(f"sample-{i}") for i in range(int(fork[2]))]
    assert used() == int(fork[4])
    refs = [int(x) for x in fork[6:fork.index("naive_blocks")]]
    assert [alloc.refcount(b) for b in prompt.table] == refs
    naive = (len(samples) + 1) * len(prompt.table)
    assert naive == int(fork[fork.index("naive_blocks") + 1])
    saved = naive - used()
    assert saved == int(fork[fork.index("saved_blocks") + 1])
    assert saved * B * KIB_PER_TOKEN_LLAMA2_7B / 1024 == float(fork[fork.index("saved_mib") + 1])
    diverge = [r for r in read_golden("cow_fork.txt") if r[0] == "diverge"]
    for row, seq in zip(diverge, samples):
        cows = seq.append_tokens(1)
        assert seq.table == [int(x) for x in row[4:row.index("cow")]]
        assert cows == int(row[-1])
    assert used() == int(rows["after"][-1])
    # the reference-counting guard
    rel = rows["release"]
    samples[0].release()
    assert alloc.refcount(0) == int(rel[rel.index("block0_refcount") + 1])
    assert (0 in alloc.free_list()) == bool(int(rel[-1]))
    for s in [prompt] + samples[1:]:
        s.release()
    assert (0 in alloc.free_list()) == bool(int(rows["release_all"][-1]))
    assert alloc.n_free == alloc.n_blocks


def test_double_free_is_refused():
    alloc = BlockAllocator(4, 16)
    b = alloc.allocate()
    assert alloc.free_block(b)
    with pytest.raises(DoubleFree):
        alloc.free_block(b)


def test_deadlock_then_preemption_example():
    rows = read_golden("deadlock_preempt.txt")
    B = int(rows[0][1])
    pool = rows[1]
    alloc = BlockAllocator(int(pool[1]), B)
    seqs = [Sequence(f"seq-{i}", alloc) for i in range(int(pool[3]))]
    for s in seqs:
        s.append_tokens(int(pool[5]))
    assert alloc.n_free == 0 and int(pool[7]) == alloc.n_blocks
    with pytest.raises(OutOfBlocks):
        seqs[0].append_tokens(1)
    assert seqs[0].n_tokens == int(pool[5])
    victim = int(rows[3][2])
    assert victim == len(seqs) - 1      # LIFO: the newest sequence is the victim
    seqs[victim].release()
    assert alloc.free_list() == [int(x) for x in rows[3][rows[3].index("free") + 1:]]
    seqs[0].append_tokens(1)
    ok = rows[4]
    assert seqs[0].table == [int(x) for x in ok[ok.index("table") + 1:ok.index("n_tokens")]]
    assert seqs[0].n_tokens == int(ok[-1])


def test_waste_never_exceeds_block_size_minus_one():
    for B in (1, 4, 8, 16, 32):
        alloc = BlockAllocator(4096, B)
        for n in range(0, 3 * B + 2):
            s = Sequence("s", alloc)
            s.append_tokens(n)
            assert 0 <= s.waste() <= B - 1
            s.release()
        assert alloc.n_free == 4096


class RecordingBatcher(ContinuousBatcher):
    """Records, at each preemption, whether the victim was the newest admission."""

    def __init__(self, *a, **k):
        super().__init__(*a, **k)
        self.victims_were_newest = []

    def _preempt_one(self, protect):
        newest = [r for r in self.running if r.rid != protect][-1]
        victim = super()._preempt_one(protect)
        self.victims_were_newest.append(victim is newest)
        return victim


@pytest.mark.parametrize("block_size,n_blocks,slots", [(16, 48, 8), (8, 96, 16), (32, 24, 6), (16, 4096, 64)])
def test_continuous_batching_trace_invariants(block_size, n_blocks, slots):
    reqs = synthetic_requests(24, seed=5, prompt_lo=32, prompt_hi=300)
    b = RecordingBatcher(reqs, slots, n_blocks, block_size)
    plans = b.run()
    # every request finished, and the caller saw each of its tokens exactly once
    for r in reqs:
        assert r.done and r.finished_at >= 0
        assert r.delivered == list(range(r.prompt_len, r.prompt_len + r.output_len))
    # the pool is whole after the drain
    assert b.alloc.n_free == b.alloc.n_blocks
    assert all(b.alloc.refcount(i) == 0 for i in range(b.alloc.n_blocks))
    for plan in plans:
        assert len(plan.rids) <= slots
        nblk = (plan.block_tables >= 0).sum(axis=1)
        waste = nblk * block_size - plan.context_lens
        assert (waste >= 0).all() and (waste <= block_size - 1).all()
        ids = plan.block_tables[plan.block_tables >= 0]
        assert len(set(ids.tolist())) == len(ids)         # no block held twice
        assert len(plan.token_row) >= len(plan.rids)
    if n_blocks < 100:
        assert b.total_preemptions > 0
        assert all(b.victims_were_newest)
    else:
        assert b.total_preemptions == 0


def replay_token_placement(plans, block_size):
    """Follow every token's label (request, position) through the plans' swap-ins,
    swap-outs and appends, in the device's order, and check that each decoded
    row finds exactly its own tokens at the slots its block table names."""
    dev, host = {}, {}
    B = block_size

    def move(src, dst, pairs):
        for a, b in pairs:
            for o in range(B):
                if (a, o) in src:
                    dst[(b, o)] = src[(a, o)]
                else:
                    dst.pop((b, o), None)

    for plan in plans:
        move(host, dev, plan.swap_in.tolist())
        move(dev, host, plan.swap_out.tolist())
        for row, pos in zip(plan.token_row.tolist(), plan.token_pos.tolist()):
            blk = int(plan.block_tables[row, pos // B])
            dev[(blk, pos % B)] = (plan.rids[row], pos)
        for b, rid in enumerate(plan.rids):
            for pos in range(int(plan.context_lens[b])):
                blk = int(plan.block_tables[b, pos // B])
                assert dev.get((blk, pos % B)) == (rid, pos), (plan.step, rid, pos)


@pytest.mark.parametrize("preempt", ["recompute", "swap"])
@pytest.mark.parametrize("block_size,n_blocks,slots", [(16, 48, 8), (8, 96, 16), (32, 24, 6)])
def test_plans_keep_every_token_in_place(preempt, block_size, n_blocks, slots):
    reqs = synthetic_requests(24, seed=5, prompt_lo=32, prompt_hi=300)
    b = ContinuousBatcher(reqs, slots, n_blocks, block_size, preempt=preempt,
                          host_blocks=4 * n_blocks)
    plans = b.run()
    assert b.total_preemptions > 0
    replay_token_placement(plans, block_size)
    for r in reqs:
        assert r.delivered == list(range(r.prompt_len, r.prompt_len + r.output_len))
    assert b.alloc.n_free == b.alloc.n_blocks
    if preempt == "swap":
        assert b.swapped_out_blocks > 0
        assert b.swapped_in_blocks == b.swapped_out_blocks
        assert b.host.n_free == b.host.n_blocks and not b.swapped
    else:
        assert all(len(p.swap_in) == 0 and len(p.swap_out) == 0 for p in plans)


def test_swap_appends_less_than_recompute():
    """Swapped-in sequences are not re-appended: the same trace appends fewer
    tokens than with recompute, and decodes the same (request, position) rows."""
    def run(mode):
        reqs = synthetic_requests(24, seed=5, prompt_lo=32, prompt_hi=300)
        b = ContinuousBatcher(reqs, 8, 48, 16, preempt=mode, host_blocks=256)
        plans = b.run()
        rows = sorted((rid, int(p.query_pos[i])) for p in plans for i, rid in enumerate(p.rids))
        return b, sum(len(p.token_row) for p in plans), rows
    rb, r_tokens, r_rows = run("recompute")
    sb, s_tokens, s_rows = run("swap")
    assert r_rows == s_rows
    assert sb.swapped_out_blocks > 0 and s_tokens < r_tokens


def test_swap_falls_back_to_recompute_when_the_host_pool_is_full():
    reqs = synthetic_requests(24, seed=5, prompt_lo=32, prompt_hi=300)
    b = ContinuousBatcher(reqs, 8, 48, 16, preempt="swap", host_blocks=1)
    plans = b.run()
    assert b.total_preemptions > 0 and b.swapped_out_blocks <= 1
    replay_token_placement(plans, 16)
    with pytest.raises(ValueError):
        ContinuousBatcher(reqs, 8, 48, 16, preempt="evict")
