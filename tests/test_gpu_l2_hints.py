"""L2 eviction priorities on the decode's K/V loads (PAGEDKV_OPT_L2_HINTS) are
a caching hint and nothing else: the decode gives bit-identical outputs with
them forced on and forced off, and those outputs match the fp64 oracle (needs
a GPU). Forced on, these small cases take the hinted loads (and the
neighbouring-sequence block-table reads that choose each block's priority)
that the automatic setting keeps for calls streaming more K/V than the L2
holds."""
import numpy as np
import pytest
import torch

import paged_kv_cache_233_gb300 as pk
from paged_support import assert_close, gpu_fill, oracle_decode, oracle_fill
from workloads import make_workload, materialize

pytestmark = pytest.mark.gpu

NEVER, ALWAYS = 1, 2


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.load()
    torch.cuda.set_device(0)
    for opt in (pk.OPT_DECODE_PATH, pk.OPT_CTAS_PER_SM, pk.OPT_STAGES, pk.OPT_L2_HINTS):
        pk.set_option(opt, 0)
    yield
    pk.set_option(pk.OPT_L2_HINTS, 0)


def bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


@pytest.mark.parametrize("dtype,Hq,Hkv,D,B,group,prefix,P", [
    ("bf16", 32, 8, 128, 16, 4, 64, 0),
    ("bf16", 32, 8, 128, 16, 4, 64, 64),
    ("bf16", 32, 8, 128, 16, 4, 64, -1),
    ("f16", 32, 32, 128, 8, 3, 32, 32),      # 8-token blocks: a hint per block box
    ("f16", 32, 32, 128, 8, 0, 0, -1),
    ("f16", 32, 32, 128, 32, 0, 0, -1),
    ("f32", 8, 4, 64, 8, 5, 48, 0),
    ("bf16", 16, 2, 64, 32, 2, 64, 64),
])
def test_hints_leave_outputs_unchanged(orc, dtype, Hq, Hkv, D, B, group, prefix, P):
    rng = np.random.default_rng(91)
    lens = rng.integers(prefix + 1, prefix + 400, size=13)
    wl = make_workload("hints", dtype, lens, Hq, Hkv, D, B, 91, prefix_group=group,
                       prefix_tokens=prefix)
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    okc, ovc, _ = oracle_fill(orc, wl, t)
    ref = oracle_decode(orc, wl, t["q"], okc, ovc)
    lens_t = torch.from_numpy(wl.context_lens).cuda()
    outs = {}
    for mode in (ALWAYS, NEVER):
        pk.set_option(pk.OPT_L2_HINTS, mode)
        out = torch.full_like(t["q"], float("nan"))
        ws = pk.new_workspace(t["q"], bt, B, P)
        pk.device_errors(reset=True)
        pk.paged_attention_decode(t["q"], kc, vc, bt, lens_t, wl.scale, out, P, ws)
        torch.cuda.synchronize()
        assert pk.device_errors() == 0
        outs[mode] = out
    pk.set_option(pk.OPT_L2_HINTS, 0)
    assert torch.equal(bits(outs[ALWAYS]), bits(outs[NEVER]))
    assert_close(outs[ALWAYS], ref, dtype, what=f"hinted loads {dtype} B={B} P={P}")


def test_hints_leave_the_shared_prefix_entry_unchanged(orc):
    B, P, prefix = 16, 64, 128
    rng = np.random.default_rng(92)
    lens = rng.integers(prefix + 1, prefix + 300, size=12)
    wl = make_workload("hints_prefix", "bf16", lens, 32, 8, 128, B, 92, prefix_group=6,
                       prefix_tokens=prefix)
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    okc, ovc, _ = oracle_fill(orc, wl, t)
    ref = oracle_decode(orc, wl, t["q"], okc, ovc)
    seq_group = torch.from_numpy(np.repeat(np.arange(2, dtype=np.int32), 6)).cuda()
    group_prefix = torch.full((2,), prefix, dtype=torch.int32, device="cuda")
    lens_t = torch.from_numpy(wl.context_lens).cuda()
    outs = {}
    for mode in (ALWAYS, NEVER):
        pk.set_option(pk.OPT_L2_HINTS, mode)
        out = torch.full_like(t["q"], float("nan"))
        pk.device_errors(reset=True)
        pk.paged_attention_decode_shared_prefix(t["q"], kc, vc, bt, lens_t, seq_group, group_prefix,
                                                wl.scale, out, P, pk.new_workspace(t["q"], bt, B, P))
        torch.cuda.synchronize()
        assert pk.device_errors() == 0
        outs[mode] = out
    pk.set_option(pk.OPT_L2_HINTS, 0)
    assert torch.equal(bits(outs[ALWAYS]), bits(outs[NEVER]))
    assert_close(outs[ALWAYS], ref, "bf16", what="shared prefix, hinted loads")
