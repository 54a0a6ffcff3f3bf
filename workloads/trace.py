"""The continuous-batching workload: a seeded scheduler run feeds the kernels.

64 requests arrive Poisson (mean 1 per step) with prompts uniform in
[32, 512] and outputs drawn from {8, 16, 32, 64, 128} (weights .3 .25 .15 .15
.15); up to `slots` of them run at once over a pool of 65,536 token slots
(4096 blocks of 16, or the same capacity at block size 8 or 32), with LIFO
preemption by recompute (or, on request, by swapping to a host pool).
Llama-2-7B layer shape: 32 heads, head_dim 128, fp16.

Every token of request r has fixed K and V rows and a fixed query row, drawn
once per request from a generator seeded by (seed, r): a preempted request
that is re-admitted re-appends exactly the bytes it had.
"""
from dataclasses import dataclass
import math

import torch

from .serving import ContinuousBatcher, synthetic_requests
from .synth import BASE_SEED, TORCH_DTYPES


@dataclass
class TraceWorkload:
    name: str
    dtype: str
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    slots: int
    requests: list
    plans: list
    max_blocks_per_seq: int
    preemptions: int
    seed: int

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def element_bytes(self):
        return 4 if self.dtype == "f32" else 2

    @property
    def torch_dtype(self):
        return TORCH_DTYPES[self.dtype]


def cb_trace(block_size=16, slots=64, pool_tokens=65536, n_requests=64, seed=BASE_SEED + 4,
             dtype="f16", n_q_heads=32, n_kv_heads=32, head_dim=128, prompt_hi=512,
             preempt="recompute", host_tokens=0):
    """The trace's step plans. preempt="swap" copies victims' blocks to a host
    pool of `host_tokens` token slots instead of recomputing them."""
    reqs = synthetic_requests(n_requests, seed=seed, prompt_hi=prompt_hi)
    n_blocks = pool_tokens // block_size
    batcher = ContinuousBatcher(reqs, slots, n_blocks, block_size, preempt=preempt,
                                host_blocks=host_tokens // block_size)
    plans = batcher.run()
    name = f"cb_trace_B{block_size}_slots{slots}" + ("_swap" if preempt == "swap" else "")
    return TraceWorkload(name, dtype, n_q_heads, n_kv_heads, head_dim, block_size, n_blocks,
                         slots, reqs, plans, batcher.max_blocks, batcher.total_preemptions, seed)


def trace_tensors(tw, device="cpu"):
    """Per-request K, V [n_req][max_tokens][Hkv][D] and Q [n_req][max_tokens][Hq][D]."""
    dev = torch.device(device)
    longest = max(r.prompt_len + r.output_len for r in tw.requests)
    dt = tw.torch_dtype
    K = torch.empty((len(tw.requests), longest, tw.n_kv_heads, tw.head_dim), dtype=dt, device=dev)
    V = torch.empty_like(K)
    Q = torch.empty((len(tw.requests), longest, tw.n_q_heads, tw.head_dim), dtype=dt, device=dev)
    for r in tw.requests:
        g = torch.Generator(device=dev)
        g.manual_seed(tw.seed * 100003 + r.rid)
        for t in (K, V, Q):
            t[r.rid] = torch.randn(t.shape[1:], generator=g, device=dev, dtype=torch.float32).to(dt)
    return {"K": K, "V": V, "Q": Q}


def step_inputs(tw, plan, tensors, device="cpu"):
    """Device tensors of one step: block tables, lengths, the appended tokens'
    (row, position) and K/V rows, and the decode queries."""
    dev = torch.device(device)
    rids = torch.tensor(plan.rids, dtype=torch.long, device=dev)
    row = torch.from_numpy(plan.token_row).to(dev)
    pos = torch.from_numpy(plan.token_pos).to(dev)
    qpos = torch.from_numpy(plan.query_pos).to(dev).long()
    tok_rid = rids[row.long()]
    return {
        "block_tables": torch.from_numpy(plan.block_tables).to(dev),
        "context_lens": torch.from_numpy(plan.context_lens).to(dev),
        "token_row": row, "token_pos": pos,
        "k": tensors["K"][tok_rid, pos.long()].contiguous(),
        "v": tensors["V"][tok_rid, pos.long()].contiguous(),
        "q": tensors["Q"][rids, qpos].contiguous(),
    }
