"""Copy-on-write block copy, CUDA path against the oracle (needs a GPU).

Random whole-block copies must be bit-exact; the serving page's fork
scenario (prompts shared by forked samples, each sample's first token
copying the shared last block into a fresh one) must leave the pools
bit-exact to the oracle's and decode every sample within tolerance.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_233_gb300 as pk
from oracle_pins import poison
from paged_support import TOL, to_f64, to_np
from workloads.serving import BlockAllocator, Sequence

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.load()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("dtype,B,Hkv,D", [("f16", 16, 32, 128), ("bf16", 8, 8, 64), ("f32", 32, 2, 64)])
def test_copy_blocks_bit_exact(orc, dtype, B, Hkv, D):
    NB = 40
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[dtype]
    g = torch.Generator(device="cuda").manual_seed(3)
    kc = torch.randn(NB, B, Hkv, D, generator=g, device="cuda").to(tdt)
    vc = torch.randn(NB, B, Hkv, D, generator=g, device="cuda").to(tdt)
    okc, ovc = to_np(kc).copy(), to_np(vc).copy()
    pairs = np.array([[0, 20], [5, 21], [7, 22], [7, 23], [3, 3], [1, NB + 4]], np.int32)
    pk.device_errors(reset=True)
    pk.paged_kv_copy_blocks(kc, vc, torch.from_numpy(pairs).cuda())
    assert pk.device_errors() & 0x02               # the out-of-pool pair was flagged
    assert orc.copy_blocks(okc, ovc, pairs) == 1
    assert to_np(kc).tobytes() == okc.tobytes() and to_np(vc).tobytes() == ovc.tobytes()


def test_fork_copy_on_write_then_decode(orc):
    """Four prompts of the Llama-2-7B layer shape, each forked into four samples."""
    B, Hkv, D, dtype = 16, 32, 128, "f16"
    rng = np.random.default_rng(12)
    alloc = BlockAllocator(256, B)
    NB = alloc.n_blocks
    gen = torch.Generator(device="cuda").manual_seed(12)
    kc = torch.full((NB, B, Hkv, D), float("nan"), dtype=torch.float16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    okc, ovc = poison(kc.shape, dtype), poison(kc.shape, dtype)

    def append(table, positions, k, v):
        bt = np.array([table], np.int32)
        seq = np.zeros(len(positions), np.int32)
        pos = np.asarray(positions, np.int32)
        sm = torch.empty(len(positions), dtype=torch.int64, device="cuda")
        pk.paged_kv_slot_mapping(torch.from_numpy(bt).cuda(), torch.from_numpy(seq).cuda(),
                                 torch.from_numpy(pos).cuda(), sm, NB, B)
        pk.paged_kv_append(k, v, sm, kc, vc)
        osm = orc.slot_mapping(bt, seq, pos, B)
        assert np.array_equal(sm.cpu().numpy(), osm)
        orc.append(to_np(k), to_np(v), osm, okc, ovc)

    seqs = []
    for p in range(4):
        prompt = Sequence(f"prompt{p}", alloc)
        n = int(rng.integers(20, 200))
        prompt.append_tokens(n)
        append(prompt.table, range(n), torch.randn(n, Hkv, D, generator=gen, device="cuda").half(),
               torch.randn(n, Hkv, D, generator=gen, device="cuda").half())
        seqs.append(prompt)
        samples = [prompt.fork(f"p{p}s{i}") for i in range(4)]
        pairs = []
        for smp in samples:
            shared_last = smp.table[-1]
            copied = smp.append_tokens(1)
            if copied:
                pairs.append([shared_last, smp.table[-1]])
        if pairs:
            pr = np.array(pairs, np.int32)
            pk.paged_kv_copy_blocks(kc, vc, torch.from_numpy(pr).cuda())
            orc.copy_blocks(okc, ovc, pr)
        for smp in samples:
            pos = smp.n_tokens - 1
            append(smp.table, [pos], torch.randn(1, Hkv, D, generator=gen, device="cuda").half(),
                   torch.randn(1, Hkv, D, generator=gen, device="cuda").half())
        seqs.extend(samples)
    assert pk.device_errors() == 0
    assert to_np(kc).tobytes() == okc.tobytes() and to_np(vc).tobytes() == ovc.tobytes()
    MB = max(len(s.table) for s in seqs)
    bt = np.full((len(seqs), MB), -1, np.int32)
    for i, s in enumerate(seqs):
        bt[i, :len(s.table)] = s.table
    lens = np.array([s.n_tokens for s in seqs], np.int32)
    q = torch.randn(len(seqs), Hkv, D, generator=gen, device="cuda").half()
    out = torch.empty_like(q)
    for P in (0, 64):
        pk.paged_attention_decode(q, kc, vc, torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda(),
                                  D ** -0.5, out, P, pk.new_workspace(q, torch.from_numpy(bt).cuda(), B, P))
        ref = orc.decode(to_np(q), okc, ovc, bt, lens, D ** -0.5, dtype)
        assert float(np.abs(to_f64(out) - ref).max()) <= TOL[dtype]
