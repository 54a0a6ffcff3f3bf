"""Allocation-free split-K decode against the fp64 oracle and against the
workspace-taking decode (needs a GPU).

paged_attention_decode_noalloc serves callers that must not allocate device
memory on their call path (a serving loop with a fixed latency budget, a
plug-in whose host application owns all device memory, a process whose free
memory belongs to another allocator): its split-K partition states live in a
fixed library-owned device array shared by every call. These tests compare
its output with the oracle and with paged_attention_decode given a caller
workspace, on calls in a row that reuse that array (fixed partitions and the
balanced split), and check that a split larger than the array is refused. The
file is named to be collected after every other test.
"""
import pytest
import torch

import paged_kv_cache_233_gb300 as pk
from paged_support import TOL, gpu_fill, oracle_decode, oracle_fill, to_f64
from workloads import make_workload, materialize

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.load()
    torch.cuda.set_device(0)
    for opt in (pk.OPT_DECODE_PATH, pk.OPT_CTAS_PER_SM, pk.OPT_STAGES):
        pk.set_option(opt, 0)


@pytest.mark.parametrize("P", [64, pk.PARTITION_BALANCED])
def test_noalloc_matches_oracle_and_workspace_decode_on_calls_in_a_row(orc, P):
    cases = [make_workload("noalloc-a", "bf16", [5, 100, 300, 777, 64], 32, 8, 128, 16, 21),
             make_workload("noalloc-b", "f16", [64, 1, 513, 40, 260, 1000], 8, 8, 64, 16, 22)]
    pk.device_errors(reset=True)
    for wl in cases:
        t = materialize(wl, "cuda")
        kc, vc, bt, _ = gpu_fill(wl, t)
        okc, ovc, _ = oracle_fill(orc, wl, t)
        lens = torch.from_numpy(wl.context_lens).cuda()
        ref = torch.empty_like(t["q"])
        pk.paged_attention_decode(t["q"], kc, vc, bt, lens, wl.scale, ref, P,
                                  pk.new_workspace(t["q"], bt, wl.block_size, P))
        # two calls in a row: the second with other queries, over the array the
        # first left behind
        q2 = (t["q"].float() * -0.75).to(t["q"].dtype)
        for q in (t["q"], q2):
            oref = oracle_decode(orc, wl, q, okc, ovc)
            out = torch.full_like(q, float("nan"))
            pk.paged_attention_decode_noalloc(q, kc, vc, bt, lens, wl.scale, out, P)
            torch.cuda.synchronize()
            assert torch.isfinite(out).all()
            err = float(abs(to_f64(out) - oref).max())
            assert err <= TOL[wl.dtype], (wl.name, P, "oracle", err)
            if q is t["q"]:
                err = (out.double() - ref.double()).abs().max().item()
                assert err <= TOL[wl.dtype], (wl.name, P, "workspace decode", err)
    assert pk.device_errors() == 0


def test_noalloc_refuses_a_split_larger_than_its_scratch():
    S, Hq, Hkv, D, B, max_blocks, P = 64, 64, 8, 128, 16, 8192, 16
    need = pk.paged_attention_workspace_bytes(S, Hq, D, max_blocks, B, P)
    assert need > pk.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(S, Hq, D, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, B, Hkv, D, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(S, max_blocks, dtype=torch.int32, device="cuda")
    lens = torch.ones(S, dtype=torch.int32, device="cuda")
    with pytest.raises(pk.PagedKVError, match="-5"):
        pk.paged_attention_decode_noalloc(q, kc, kc, bt, lens, 0.1, torch.empty_like(q), P)
