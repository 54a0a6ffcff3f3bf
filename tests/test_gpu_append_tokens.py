"""paged_kv_append_tokens (slot mapping and append in one launch) against the
oracle and against the two separate calls (needs a GPU)."""
import numpy as np
import pytest
import torch

import paged_kv_cache_233_gb300 as pk
from paged_support import oracle_fill, to_np
from workloads import make_workload, materialize, new_pools, preset

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.load()
    torch.cuda.set_device(0)


def fused_fill(wl, t, with_slots):
    kc, vc = new_pools(wl, "cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    slots = {}
    for tag, seq, pos, k, v in (("fill", wl.fill_seq, wl.fill_pos, t["k_fill"], t["v_fill"]),
                                ("step", wl.step_seq, wl.step_pos, t["k_step"], t["v_step"])):
        sm = torch.full((len(seq),), 12345, dtype=torch.int64, device="cuda") if with_slots else None
        if len(seq):
            pk.paged_kv_append_tokens(k, v, bt, torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda(),
                                      kc, vc, slot_mapping=sm)
        slots[tag] = sm
    return kc, vc, slots


@pytest.mark.parametrize("wl_name", ["tiny", "smoke_bf16", "mha_rows", "odd_rows"])
@pytest.mark.parametrize("with_slots", [True, False])
def test_pools_and_slots_bit_exact_to_the_oracle(orc, wl_name, with_slots):
    if wl_name == "tiny":
        wl = preset("tiny")
    elif wl_name == "smoke_bf16":
        wl = make_workload("fused_bf16", "bf16", [1, 17, 40, 300], 32, 8, 128, 16, 41)
    elif wl_name == "mha_rows":
        wl = make_workload("fused_mha", "f16", [5, 130, 700, 64], 32, 32, 128, 8, 42)
    else:
        # 384-byte rows (3 kv heads x 64 x fp16): 24 chunks of 16 bytes for a
        # row's 32 threads, so some threads of every row copy nothing
        wl = make_workload("fused_odd", "f16", [3, 50, 17, 129], 6, 3, 64, 16, 44)
    t = materialize(wl, "cuda")
    pk.device_errors(reset=True)
    kc, vc, slots = fused_fill(wl, t, with_slots)
    torch.cuda.synchronize()
    assert pk.device_errors() == 0
    okc, ovc, oslots = oracle_fill(orc, wl, t)
    assert to_np(kc).tobytes() == okc.tobytes()
    assert to_np(vc).tobytes() == ovc.tobytes()
    if with_slots:
        for tag in ("fill", "step"):
            assert np.array_equal(slots[tag].cpu().numpy(), oslots[tag])


def test_padding_and_bad_tokens_match_the_separate_calls():
    """Padding, a sequence index out of range, a position past the table and a
    block id outside the pool: the same slots, pools and error bits as
    paged_kv_slot_mapping followed by paged_kv_append."""
    wl = make_workload("fused_bad", "f16", [20, 40], 4, 2, 64, 16, 43)
    t = materialize(wl, "cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    bt_bad = bt.clone()
    bt_bad[1, 0] = wl.num_blocks + 3               # a block id outside the pool
    seq = torch.tensor([0, 0, 1, 5, 0, 1, -1], dtype=torch.int32, device="cuda")
    pos = torch.tensor([3, -1, 2, 0, 10 ** 6, 7, 1], dtype=torch.int32, device="cuda")
    k = torch.randn(7, 2, 64, device="cuda").half()
    v = torch.randn(7, 2, 64, device="cuda").half()
    results = []
    for fused in (False, True):
        kc, vc = new_pools(wl, "cuda")
        sm = torch.full((7,), 12345, dtype=torch.int64, device="cuda")
        pk.device_errors(reset=True)
        for table in (bt, bt_bad):
            if fused:
                pk.paged_kv_append_tokens(k, v, table, seq, pos, kc, vc, slot_mapping=sm)
            else:
                pk.paged_kv_slot_mapping(table, seq, pos, sm, wl.num_blocks, wl.block_size)
                pk.paged_kv_append(k, v, sm, kc, vc)
        torch.cuda.synchronize()
        results.append((to_np(kc).tobytes(), to_np(vc).tobytes(), sm.cpu().numpy(),
                        pk.device_errors()))
    (k0, v0, s0, e0), (k1, v1, s1, e1) = results
    assert k0 == k1 and v0 == v1
    assert np.array_equal(s0, s1)
    assert e0 == e1 and e0 != 0
    # padding, the bad sequence, the position past the table and the bad block are all -1
    assert (s1[[1, 3, 4, 6]] == -1).all()
