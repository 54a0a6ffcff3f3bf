"""Shared plumbing for the GPU parity tests: build one workload's pools and
outputs on both sides from the same seeded inputs.

GPU side: the library's slot mapping + append fill NaN-poisoned device
pools, then the library's decode runs. Oracle side: the oracle's slot mapping
+ append fill NaN-poisoned host pools, then the oracle decodes. The two sides
share only the workload description and the drawn q/k/v values.
"""
import numpy as np
import torch

import paged_kv_cache_233_gb300 as pk
from workloads import materialize, new_pools

TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 1.5e-2}


def to_np(t):
    """Host copy of a tensor as the oracle reads it (bf16 as uint16 bits)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def to_f64(t):
    return t.detach().cpu().double().numpy()


def gpu_fill(wl, tensors, device="cuda"):
    """Device pools filled through paged_kv_slot_mapping + paged_kv_append."""
    kc, vc = new_pools(wl, device)
    bt = torch.from_numpy(wl.block_tables).to(device)
    slots = {}
    for tag, seq, pos, k, v in (("fill", wl.fill_seq, wl.fill_pos, tensors["k_fill"], tensors["v_fill"]),
                                ("step", wl.step_seq, wl.step_pos, tensors["k_step"], tensors["v_step"])):
        n = len(seq)
        sm = torch.empty(n, dtype=torch.int64, device=device)
        if n:
            pk.paged_kv_slot_mapping(bt, torch.from_numpy(seq).to(device),
                                     torch.from_numpy(pos).to(device), sm, wl.num_blocks,
                                     wl.block_size)
            pk.paged_kv_append(k, v, sm, kc, vc)
        slots[tag] = sm
    return kc, vc, bt, slots


def gpu_decode(wl, q, kc, vc, bt, partition_tokens=0, device="cuda"):
    lens = torch.from_numpy(wl.context_lens).to(device)
    out = torch.full_like(q, float("nan"))
    ws = pk.new_workspace(q, bt, wl.block_size, partition_tokens)
    pk.paged_attention_decode(q, kc, vc, bt, lens, wl.scale, out, partition_tokens, ws)
    return out, ws


def oracle_fill(orc, wl, tensors):
    """Host pools filled through the oracle's slot mapping + append."""
    from oracle_pins import poison
    shape = (wl.num_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim)
    kc, vc = poison(shape, wl.dtype), poison(shape, wl.dtype)
    slots = {}
    for tag, seq, pos, k, v in (("fill", wl.fill_seq, wl.fill_pos, tensors["k_fill"], tensors["v_fill"]),
                                ("step", wl.step_seq, wl.step_pos, tensors["k_step"], tensors["v_step"])):
        sm = orc.slot_mapping(wl.block_tables, seq, pos, wl.block_size)
        bad = orc.append(to_np(k), to_np(v), sm, kc, vc)
        assert bad == 0
        slots[tag] = sm
    return kc, vc, slots


def oracle_decode(orc, wl, q, kc, vc, units=None):
    return orc.decode(to_np(q), kc, vc, wl.block_tables, wl.context_lens, wl.scale, wl.dtype,
                      units=units)


def assert_close(got, ref, dtype, rows=None, what=""):
    """Max-abs error over the given (seq, q head) rows (all rows by default)."""
    g = to_f64(got)
    if rows is not None:
        g = np.stack([g[s, h] for s, h in rows])
        ref = np.stack([ref[s, h] for s, h in rows])
    assert np.isfinite(g).all(), f"{what}: non-finite outputs"
    err = float(np.abs(g - ref).max()) if g.size else 0.0
    assert err <= TOL[dtype], f"{what}: max-abs error {err:.3e} > {TOL[dtype]:.1e}"
    return err


def units_to_rows(wl, units):
    g = wl.group
    return [(s, h * g + j) for s, h in units for j in range(g)]
