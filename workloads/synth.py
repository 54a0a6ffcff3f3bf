"""Seeded synthetic paged-KV workloads (lengths, block tables, token lists, q/k/v).

A workload describes one decode step of one layer:

* ``context_lens[s]`` tokens of sequence ``s`` are attended over in the step;
  the step's own new token is the last of them (position ``L_s - 1``);
* ``block_tables[s]`` lists the physical blocks the allocator gave sequence
  ``s``, in logical order (``ceil(L_s / B)`` of them, unused entries ``-1``);
* ``fill_seq/fill_pos`` are the tokens already in the cache before the step
  (a shared prefix is written once, by its group's first sequence);
* ``step_seq/step_pos`` are the step's new tokens, one per sequence.

Both sides build their pools from these lists through their own slot
mapping and append, so nothing here decides where a token's bytes live.
Values of q, k and v are drawn N(0, 1) in fp32 from a seeded torch generator
and rounded to the workload's element type.
"""
from dataclasses import dataclass, field
import math

import numpy as np
import torch

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}

BASE_SEED = 7


@dataclass
class PagedWorkload:
    name: str
    dtype: str
    num_seqs: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    context_lens: np.ndarray
    block_tables: np.ndarray
    fill_seq: np.ndarray
    fill_pos: np.ndarray
    step_seq: np.ndarray
    step_pos: np.ndarray
    seed: int
    scale: float
    partition_tokens: int = 0
    groups: list = field(default_factory=list)
    prefix_blocks: int = 0

    @property
    def max_blocks_per_seq(self):
        return int(self.block_tables.shape[1])

    @property
    def group(self):
        return self.n_q_heads // self.n_kv_heads

    @property
    def torch_dtype(self):
        return TORCH_DTYPES[self.dtype]

    @property
    def element_bytes(self):
        return 4 if self.dtype == "f32" else 2

    @property
    def row_bytes(self):
        """Bytes of one token's K (or V) row: n_kv_heads * head_dim elements."""
        return self.n_kv_heads * self.head_dim * self.element_bytes

    def blocks_in_use(self):
        """Distinct physical blocks referenced by the block tables."""
        bt = self.block_tables
        return np.unique(bt[bt >= 0])

    def refcounts(self):
        """How many sequences reference each physical block."""
        rc = np.zeros(self.num_blocks, dtype=np.int64)
        for s in range(self.num_seqs):
            ids = self.block_tables[s][self.block_tables[s] >= 0]
            np.add.at(rc, ids, 1)
        return rc


def _blocks_for(length, block_size):
    """Blocks a sequence of `length` tokens holds: the allocator grows one
    block at a time, so it holds ceil(length / block_size) of them."""
    return -(-int(length) // block_size)


def make_workload(name, dtype, lens, n_q_heads, n_kv_heads, head_dim, block_size, seed,
                  pool_factor=1.25, num_blocks=None, prefix_group=0, prefix_tokens=0,
                  partition_tokens=0, table_pad=0):
    """Build a workload from decode lengths `lens` (the step token included).

    Physical block ids come from one seeded permutation of the pool, taken in
    order: each prefix group's shared blocks once, then every sequence's
    private blocks. `prefix_group` sequences in a row share their first
    `prefix_tokens` tokens (a whole number of blocks, strictly shorter than
    each member's length so that the step never writes into a shared block).
    """
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int64)
    S = int(lens.shape[0])
    B = int(block_size)
    if n_q_heads % n_kv_heads:
        raise ValueError("n_q_heads must be a multiple of n_kv_heads")
    need = np.array([_blocks_for(L, B) for L in lens], dtype=np.int64)
    groups = []
    prefix_blocks = 0
    if prefix_group > 1 and prefix_tokens > 0:
        if prefix_tokens % B:
            raise ValueError("a shared prefix must be a whole number of blocks")
        prefix_blocks = prefix_tokens // B
        groups = [list(range(g0, min(g0 + prefix_group, S))) for g0 in range(0, S, prefix_group)]
        for grp in groups:
            if min(int(lens[s]) for s in grp) <= prefix_tokens:
                raise ValueError("every group member must extend past the shared prefix")
    unique_need = int(need.sum()) - sum(prefix_blocks * (len(g) - 1) for g in groups)
    NB = int(num_blocks) if num_blocks is not None else int(math.ceil(pool_factor * unique_need))
    if NB < unique_need:
        raise ValueError("pool too small for the workload")
    perm = rng.permutation(NB).astype(np.int32)
    take = iter(perm.tolist())
    MB = int(need.max()) + int(table_pad) if S else 1
    bt = np.full((S, MB), -1, dtype=np.int32)
    leader_of = {}
    for grp in groups:
        shared = [next(take) for _ in range(prefix_blocks)]
        for s in grp:
            bt[s, :prefix_blocks] = shared
            leader_of[s] = grp[0]
    for s in range(S):
        first = prefix_blocks if s in leader_of else 0
        for j in range(first, int(need[s])):
            bt[s, j] = next(take)
    fill_seq, fill_pos = [], []
    for s in range(S):
        L = int(lens[s])
        start = prefix_tokens if (s in leader_of and leader_of[s] != s) else 0
        fill_seq.append(np.full(max(L - 1 - start, 0), s, dtype=np.int32))
        fill_pos.append(np.arange(start, max(L - 1, start), dtype=np.int32))
    step_mask = lens > 0
    step_seq = np.nonzero(step_mask)[0].astype(np.int32)
    step_pos = (lens[step_mask] - 1).astype(np.int32)
    return PagedWorkload(
        name=name, dtype=dtype, num_seqs=S, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads,
        head_dim=head_dim, block_size=B, num_blocks=NB,
        context_lens=lens.astype(np.int32), block_tables=bt,
        fill_seq=np.concatenate(fill_seq) if fill_seq else np.zeros(0, np.int32),
        fill_pos=np.concatenate(fill_pos) if fill_pos else np.zeros(0, np.int32),
        step_seq=step_seq, step_pos=step_pos, seed=int(seed),
        scale=1.0 / math.sqrt(head_dim), partition_tokens=int(partition_tokens),
        groups=groups, prefix_blocks=prefix_blocks)


# ---------------------------------------------------------------------------
# The five named workloads. Index i uses seed BASE_SEED + i.
# ---------------------------------------------------------------------------

def tiny(seed=BASE_SEED + 0):
    """4 sequences that held {1, 17, 33, 64} tokens and each append one more:
    decode over {2, 18, 34, 65} tokens; B = 16, pool of 32 blocks; 4 q heads,
    2 kv heads, head_dim 64, fp32."""
    before = np.array([1, 17, 33, 64])
    return make_workload("tiny", "f32", before + 1, 4, 2, 64, 16, seed, num_blocks=32)


def mha7b(seed=BASE_SEED + 1, num_seqs=64, lo=128, hi=2048):
    """Llama-2-7B-shaped MHA layer: 32 q = 32 kv heads, head_dim 128, fp16,
    B = 16, lengths uniform in [128, 2048], pool 1.25x the need, shuffled."""
    rng = np.random.default_rng(seed + 1000)
    lens = rng.integers(lo, hi, size=num_seqs, endpoint=True)
    return make_workload("mha7b", "f16", lens, 32, 32, 128, 16, seed)


def gqa8b_prefix(seed=BASE_SEED + 2, num_seqs=256, median=1024, sigma=0.75, cap=8192,
                 prefix_tokens=512, group=16):
    """Llama-3-8B-shaped GQA layer with prefix sharing: 32 q / 8 kv heads,
    head_dim 128, bf16, B = 16; log-normal lengths (median 1024, sigma 0.75)
    clipped to [prefix + 1, 8192]; groups of 16 share a 512-token prefix."""
    rng = np.random.default_rng(seed + 1000)
    lens = np.rint(rng.lognormal(math.log(median), sigma, size=num_seqs))
    lens = np.clip(lens, prefix_tokens + 1, cap).astype(np.int64)
    return make_workload("gqa8b_prefix", "bf16", lens, 32, 8, 128, 16, seed,
                         prefix_group=group, prefix_tokens=prefix_tokens)


def longctx_splitk(seed=BASE_SEED + 3, num_seqs=8, lo=32768, hi=131072):
    """Long-context layer: 64 q / 8 kv heads, head_dim 128, bf16, B = 16,
    lengths uniform in [32768, 131072], shuffled; 512-token partitions."""
    rng = np.random.default_rng(seed + 1000)
    lens = rng.integers(lo, hi, size=num_seqs, endpoint=True)
    return make_workload("longctx_splitk", "bf16", lens, 64, 8, 128, 16, seed,
                         partition_tokens=512)


def chunked_prefill(name, dtype, before, chunk, n_q_heads, n_kv_heads, head_dim, block_size,
                    seed, **kw):
    """One chunked-prefill step: sequence s holds `before[s]` cached tokens and
    appends a chunk of `chunk[s]` tokens whose rows then attend. The workload's
    lengths count the chunk (every token, the chunk included, is filled into the
    pools); query_start delimits each sequence's chunk rows."""
    before = np.asarray(before, dtype=np.int64)
    chunk = np.asarray(chunk, dtype=np.int64)
    wl = make_workload(name, dtype, before + chunk, n_q_heads, n_kv_heads, head_dim, block_size,
                       seed, **kw)
    query_start = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
    return wl, query_start


def prefill_mha7b(seed=BASE_SEED + 5, num_seqs=16, chunk=512, max_before=3584):
    """Llama-2-7B-shaped MHA layer (32 heads, head_dim 128, fp16, B = 16): 16
    sequences each append a 512-token chunk after U[0, 3584] cached tokens."""
    rng = np.random.default_rng(seed + 1000)
    before = rng.integers(0, max_before, size=num_seqs, endpoint=True)
    return chunked_prefill("prefill_mha7b", "f16", before, np.full(num_seqs, chunk), 32, 32, 128,
                           16, seed)


def prefill_queries(wl, query_start, device="cpu"):
    """Query rows [num_tokens][n_q_heads][head_dim] of a chunked-prefill step, N(0, 1)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(wl.seed) + 500)
    n = int(query_start[-1])
    return torch.randn((n, wl.n_q_heads, wl.head_dim), generator=gen, device=dev,
                       dtype=torch.float32).to(wl.torch_dtype)


def subset(wl, seqs):
    """The same workload restricted to sequences `seqs` (renumbered 0..k-1):
    their lengths, block-table rows and tokens, in the same pool. A shared
    prefix is written by the first kept member of its group."""
    seqs = [int(s) for s in seqs]
    keep = {s: i for i, s in enumerate(seqs)}
    prefix_tokens = wl.prefix_blocks * wl.block_size
    writer = {}
    groups = []
    for grp in wl.groups:
        kept = [s for s in grp if s in keep]
        for s in kept:
            writer[s] = kept[0]
        if len(kept) > 1:
            groups.append([keep[s] for s in kept])
    fill_seq, fill_pos = [], []
    for s in seqs:
        L = int(wl.context_lens[s])
        start = prefix_tokens if writer.get(s, s) != s else 0
        fill_seq.append(np.full(max(L - 1 - start, 0), keep[s], dtype=np.int32))
        fill_pos.append(np.arange(start, max(L - 1, start), dtype=np.int32))
    lens = wl.context_lens[seqs].astype(np.int32)
    step_mask = lens > 0
    return PagedWorkload(
        name=f"{wl.name}[{len(seqs)} of {wl.num_seqs} seqs]", dtype=wl.dtype, num_seqs=len(seqs),
        n_q_heads=wl.n_q_heads, n_kv_heads=wl.n_kv_heads, head_dim=wl.head_dim,
        block_size=wl.block_size, num_blocks=wl.num_blocks, context_lens=lens,
        block_tables=wl.block_tables[seqs].copy(),
        fill_seq=np.concatenate(fill_seq) if fill_seq else np.zeros(0, np.int32),
        fill_pos=np.concatenate(fill_pos) if fill_pos else np.zeros(0, np.int32),
        step_seq=np.nonzero(step_mask)[0].astype(np.int32),
        step_pos=(lens[step_mask] - 1).astype(np.int32), seed=wl.seed, scale=wl.scale,
        partition_tokens=wl.partition_tokens, groups=groups,
        prefix_blocks=wl.prefix_blocks if groups else 0)


PRESETS = {"tiny": tiny, "mha7b": mha7b, "gqa8b_prefix": gqa8b_prefix,
           "longctx_splitk": longctx_splitk}


def preset(name, **overrides):
    return PRESETS[name](**overrides)


# ---------------------------------------------------------------------------
# Tensors.
# ---------------------------------------------------------------------------

def materialize(wl, device="cpu", chunk_tokens=1 << 16):
    """q [S][Hq][D], k/v_fill [T][Hkv][D], k/v_step [S'][Hkv][D], drawn N(0, 1)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(wl.seed))
    dt = wl.torch_dtype

    def draw(rows, row_shape):
        out = torch.empty((rows,) + row_shape, dtype=dt, device=dev)
        for r0 in range(0, rows, chunk_tokens):
            r1 = min(rows, r0 + chunk_tokens)
            out[r0:r1] = torch.randn((r1 - r0,) + row_shape, generator=gen, device=dev,
                                     dtype=torch.float32).to(dt)
        return out

    kv_row = (wl.n_kv_heads, wl.head_dim)
    q = draw(wl.num_seqs, (wl.n_q_heads, wl.head_dim))
    k_fill = draw(len(wl.fill_seq), kv_row)
    v_fill = draw(len(wl.fill_seq), kv_row)
    k_step = draw(len(wl.step_seq), kv_row)
    v_step = draw(len(wl.step_seq), kv_row)
    return {"q": q, "k_fill": k_fill, "v_fill": v_fill, "k_step": k_step, "v_step": v_step}


def new_pools(wl, device="cpu", fill=float("nan")):
    """Fresh K and V pools [num_blocks][block_size][n_kv_heads][head_dim],
    poisoned with `fill` so that any slot nobody wrote shows up if read."""
    shape = (wl.num_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim)
    k = torch.full(shape, fill, dtype=wl.torch_dtype, device=device)
    v = torch.full(shape, fill, dtype=wl.torch_dtype, device=device)
    return k, v
