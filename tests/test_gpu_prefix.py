"""Shared-prefix decode against the fp64 oracle (needs a GPU).

paged_attention_decode_shared_prefix must give what paged_attention_decode
gives (the oracle, within the dtype's tolerance) while reading each shared
prefix partition once per chunk of group members.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_233_gb300 as pk
from paged_support import TOL, assert_close, gpu_fill, oracle_decode, oracle_fill, to_np
from workloads import make_workload, materialize, preset

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.load()
    torch.cuda.set_device(0)
    for opt in (pk.OPT_DECODE_PATH, pk.OPT_CTAS_PER_SM, pk.OPT_STAGES):
        pk.set_option(opt, 0)


def group_arrays(wl, prefix=None):
    seq_group = np.full(wl.num_seqs, -1, np.int32)
    for gi, grp in enumerate(wl.groups):
        seq_group[grp] = gi
    pre = np.full(len(wl.groups), wl.prefix_blocks * wl.block_size if prefix is None else prefix,
                  np.int32)
    return torch.from_numpy(seq_group).cuda(), torch.from_numpy(pre).cuda()


def shared_decode(wl, t, kc, vc, bt, P, seq_group, group_prefix):
    lens = torch.from_numpy(wl.context_lens).cuda()
    out = torch.full_like(t["q"], float("nan"))
    ws = pk.new_workspace(t["q"], bt, wl.block_size, P)
    pk.paged_attention_decode_shared_prefix(t["q"], kc, vc, bt, lens, seq_group, group_prefix,
                                            wl.scale, out, P, ws)
    return out


@pytest.mark.parametrize("dtype,Hq,Hkv,D,group,prefix,P", [
    ("bf16", 32, 8, 128, 16, 512, 256),     # the GQA workload's shape: 2 members per chunk
    ("f16", 32, 32, 128, 8, 256, 128),      # MHA: 8 members fill the tile
    ("bf16", 16, 4, 64, 5, 96, 32),         # odd group size, D 64
    ("bf16", 64, 8, 128, 4, 512, 512),      # group of 8 q heads: one member per chunk
    ("f32", 8, 4, 64, 3, 64, 32),           # CUDA-core path: one member per chunk
    ("bf16", 32, 8, 128, 12, 512, 256),     # runs of 12 (sequences 24-35 straddle the set-up
                                            # scan's 32-sequence chunks): 2 members per chunk
    ("f16", 32, 32, 128, 11, 256, 128),     # runs of 11 (22-32 straddle them): 8 members per chunk
])
def test_shared_prefix_matches_oracle(orc, dtype, Hq, Hkv, D, group, prefix, P):
    rng = np.random.default_rng(7)
    lens = rng.integers(prefix + 1, prefix + 700, size=group * 3)
    wl = make_workload("shared", dtype, lens, Hq, Hkv, D, 16, 71, prefix_group=group,
                       prefix_tokens=prefix)
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    okc, ovc, _ = oracle_fill(orc, wl, t)
    ref = oracle_decode(orc, wl, t["q"], okc, ovc)
    sg, gp = group_arrays(wl)
    pk.device_errors(reset=True)
    out = shared_decode(wl, t, kc, vc, bt, P, sg, gp)
    assert pk.device_errors() == 0
    assert_close(out, ref, dtype, what=f"shared prefix {dtype} g={Hq // Hkv}")


def test_shared_prefix_edge_cases(orc):
    """Prefixes that are not a whole number of partitions, members decoded over
    exactly the prefix or less than one partition, ungrouped sequences in
    between, and a group of one."""
    B, P = 16, 64
    lens = [300, 300, 300, 300, 300, 300, 300]
    wl = make_workload("edge", "f16", lens, 32, 32, 128, B, 72, prefix_group=3, prefix_tokens=160)
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    okc, ovc, _ = oracle_fill(orc, wl, t)
    # decode over fewer tokens than written (all inside the written tokens): member
    # 2 of group 0 over exactly its one-partition prefix, member 0 of group 1 over
    # 160 tokens of which 150 are declared shared (two whole partitions)
    wl.context_lens = np.array([300, 160, 64, 250, 160, 299, 80], np.int32)
    seq_group = np.array([0, 0, 0, -1, 1, 1, 2], np.int32)
    group_prefix = np.array([64, 150, 64], np.int32)
    # sequence 6 (group 2, alone) shares nothing real, so its prefix is its own tokens
    ref = oracle_decode(orc, wl, t["q"], okc, ovc)
    lens_t = torch.from_numpy(wl.context_lens).cuda()
    out = torch.full_like(t["q"], float("nan"))
    pk.device_errors(reset=True)
    pk.paged_attention_decode_shared_prefix(
        t["q"], kc, vc, bt, lens_t, torch.from_numpy(seq_group).cuda(),
        torch.from_numpy(group_prefix).cuda(), wl.scale, out, P, pk.new_workspace(t["q"], bt, B, P))
    assert pk.device_errors() == 0
    assert_close(out, ref, "f16", what="shared prefix edges")


def test_prefix_longer_than_a_member_is_flagged():
    wl = make_workload("bad", "bf16", [100, 100], 8, 4, 64, 16, 73)
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    pk.device_errors(reset=True)
    sg = torch.tensor([0, 0], dtype=torch.int32, device="cuda")
    gp = torch.tensor([128], dtype=torch.int32, device="cuda")
    out = shared_decode(wl, t, kc, vc, bt, 32, sg, gp)
    torch.cuda.synchronize()
    assert pk.device_errors() & 0x04


def test_group_id_past_the_groups_is_flagged(orc):
    """A group id outside [0, num_groups) sets the sequence-index bit and that
    sequence is decoded on its own, as by plain decode."""
    wl = make_workload("badgroup", "bf16", [100, 100, 70], 8, 4, 64, 16, 74)
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    okc, ovc, _ = oracle_fill(orc, wl, t)
    ref = oracle_decode(orc, wl, t["q"], okc, ovc)
    pk.device_errors(reset=True)
    sg = torch.tensor([0, 5, -1], dtype=torch.int32, device="cuda")
    gp = torch.tensor([0], dtype=torch.int32, device="cuda")
    out = shared_decode(wl, t, kc, vc, bt, 32, sg, gp)
    torch.cuda.synchronize()
    assert pk.device_errors() == 0x10
    assert_close(out, ref, "bf16", what="group id past the groups")


@pytest.mark.parametrize("bad", [5, -5])
def test_bad_group_id_inside_a_prefix_group(orc, bad):
    """A bad group id (past the groups, or negative other than -1) between the
    members of a group whose prefix spans several partitions: the bad sequence
    is flagged and decoded on its own, the members after it start a new run of
    the group, and every output matches the oracle."""
    B, P, prefix = 16, 32, 96
    lens = [200, 150, 180, 170, 300]
    wl = make_workload("badmember", "bf16", lens, 32, 8, 128, B, 75, prefix_group=5,
                       prefix_tokens=prefix)
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    okc, ovc, _ = oracle_fill(orc, wl, t)
    ref = oracle_decode(orc, wl, t["q"], okc, ovc)
    pk.device_errors(reset=True)
    sg = torch.tensor([0, bad, 0, 0, 0], dtype=torch.int32, device="cuda")
    gp = torch.tensor([prefix], dtype=torch.int32, device="cuda")
    out = shared_decode(wl, t, kc, vc, bt, P, sg, gp)
    torch.cuda.synchronize()
    assert pk.device_errors() == 0x10
    assert_close(out, ref, "bf16", what=f"group id {bad} inside a prefix group")


def test_gqa_prefix_workload_full_size(orc):
    """The GQA batch-256 workload with its 16-member, 512-token prefix groups."""
    wl = preset("gqa8b_prefix")
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    sg, gp = group_arrays(wl)
    out = shared_decode(wl, t, kc, vc, bt, 320, sg, gp)
    plain = torch.empty_like(out)
    pk.paged_attention_decode(t["q"], kc, vc, bt, torch.from_numpy(wl.context_lens).cuda(), wl.scale,
                              plain, 320, pk.new_workspace(t["q"], bt, wl.block_size, 320))
    assert float((out.double() - plain.double()).abs().max()) <= TOL["bf16"]
    # the oracle decodes its own pools (its slot mapping + append of the same
    # tokens), and the GPU's pools equal them byte for byte
    okc, ovc, _ = oracle_fill(orc, wl, t)
    assert to_np(kc).view(np.uint8).tobytes() == okc.view(np.uint8).tobytes()
    assert to_np(vc).view(np.uint8).tobytes() == ovc.view(np.uint8).tobytes()
    units = [(s, h) for s in (0, 1, 15, 16, 100, 255) for h in (0, 7)]
    ref = oracle_decode(orc, wl, t["q"], okc, ovc, units=units)
    rows = [(s, h * 4 + j) for s, h in units for j in range(4)]
    assert_close(out, ref, "bf16", rows=rows, what="gqa prefix full size")
