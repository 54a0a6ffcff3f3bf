"""The C ABI library loads and exports what include/pagedkv.h declares (CPU only).

No call here reaches the GPU: only host-side argument checks, which return
before anything is enqueued, and pure size arithmetic.
"""
import ctypes
import os
import re

import pytest

import paged_kv_cache_233_gb300 as pk
from paged_kv_cache_233_gb300 import build as pk_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "pagedkv.h")

INVALID, UNSUPPORTED, WORKSPACE = -1, -2, -5


@pytest.fixture(scope="module")
def lib():
    pk_build.build()
    return pk.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*([a-z_0-9]+)\s*\(", text,
                                 flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for name in ("paged_kv_slot_mapping", "paged_kv_append", "paged_attention_decode",
                 "paged_attention_workspace_bytes", "pagedkv_status_string"):
        assert name in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(pk.library_path())
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared in pagedkv.h but not exported"


def test_abi_version_and_status_strings(lib):
    assert pk.abi_version() == 1
    assert pk.status_string(0) == "ok"
    for st in (-1, -2, -3, -4, -5):
        assert pk.status_string(st) and pk.status_string(st) != "unknown status"
    assert pk.status_string(12345) == "unknown status"


def _decode(lib, **kw):
    args = dict(q=1 << 12, k=1 << 12, v=1 << 12, bt=1 << 12, lens=1 << 12, scale=0.125, out=1 << 12,
                S=4, Hq=4, Hkv=2, D=64, NB=32, B=16, MB=5, P=0, ws=None, ws_bytes=0, dtype=0)
    args.update(kw)
    return lib.paged_attention_decode(
        ctypes.c_void_p(args["q"]), ctypes.c_void_p(args["k"]), ctypes.c_void_p(args["v"]),
        ctypes.c_void_p(args["bt"]), ctypes.c_void_p(args["lens"]), args["scale"],
        ctypes.c_void_p(args["out"]), args["S"], args["Hq"], args["Hkv"], args["D"], args["NB"],
        args["B"], args["MB"], args["P"], ctypes.c_void_p(args["ws"]), args["ws_bytes"],
        args["dtype"], None)


def test_decode_rejects_bad_arguments_on_the_host(lib):
    assert _decode(lib, Hq=3, Hkv=2) == INVALID
    assert _decode(lib, D=96) == UNSUPPORTED
    assert _decode(lib, B=12) == UNSUPPORTED
    assert _decode(lib, Hq=32, Hkv=2) == UNSUPPORTED        # group of 16
    assert _decode(lib, P=100) == INVALID                    # not a multiple of 16
    assert _decode(lib, dtype=7) == INVALID
    assert _decode(lib, scale=float("nan")) == INVALID
    assert _decode(lib, q=(1 << 12) + 8) == INVALID          # misaligned
    assert _decode(lib, out=0) == INVALID                    # null
    assert _decode(lib, P=16, ws=None) == WORKSPACE
    assert _decode(lib, P=-1, ws=None) == WORKSPACE          # balanced split needs a workspace
    assert _decode(lib, P=-2) == INVALID
    assert _decode(lib, P=16, ws=1 << 12, ws_bytes=64) == WORKSPACE
    assert _decode(lib, S=0) == 0                            # nothing to do, nothing enqueued
    assert _decode(lib, S=5000) == UNSUPPORTED


def test_append_and_slot_mapping_reject_bad_arguments(lib):
    vp = ctypes.c_void_p
    # row of 3 heads x 2 fp16 = 12 bytes is not a multiple of 16
    assert lib.paged_kv_append(vp(16), vp(16), vp(16), vp(16), vp(16), 4, 8, 16, 3, 2, 1, None) == INVALID
    assert lib.paged_kv_append(vp(16), vp(16), vp(16), vp(16), vp(16), 4, 8, 16, 2, 64, 9, None) == INVALID
    assert lib.paged_kv_append(vp(0), vp(0), vp(0), vp(0), vp(0), 0, 8, 16, 2, 64, 1, None) == 0
    assert lib.paged_kv_append(vp(0), vp(16), vp(16), vp(16), vp(16), 4, 8, 16, 2, 64, 1, None) == INVALID
    assert lib.paged_kv_slot_mapping(vp(16), vp(16), vp(16), vp(16), 4, 2, 0, 16, 8, None) == INVALID
    assert lib.paged_kv_slot_mapping(vp(0), vp(0), vp(0), vp(0), 0, 2, 4, 16, 8, None) == 0


def test_append_tokens_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p

    def call(**kw):
        a = dict(k=16, v=16, bt=16, seq=16, pos=16, sm=None, kc=16, vc=16, T=4, S=2, MB=4, NB=8,
                 B=16, H=2, D=64, dtype=1)
        a.update(kw)
        return lib.paged_kv_append_tokens(vp(a["k"]), vp(a["v"]), vp(a["bt"]), vp(a["seq"]),
                                          vp(a["pos"]), vp(a["sm"]), vp(a["kc"]), vp(a["vc"]),
                                          a["T"], a["S"], a["MB"], a["NB"], a["B"], a["H"], a["D"],
                                          a["dtype"], None)

    assert call(T=-1) == INVALID
    assert call(MB=0) == INVALID
    assert call(NB=0) == INVALID
    assert call(dtype=9) == INVALID
    assert call(H=3, D=2) == INVALID                 # 12-byte rows
    assert call(k=24) == INVALID                     # misaligned K rows
    assert call(bt=18) == INVALID                    # misaligned block table
    assert call(sm=20) == INVALID                    # misaligned slot output
    assert call(seq=0) == INVALID                    # no token_seq
    assert call(T=0, k=0, v=0, bt=0, seq=0, pos=0, kc=0, vc=0) == 0   # nothing to do


def test_swap_and_copy_blocks_reject_bad_arguments(lib):
    vp = ctypes.c_void_p
    # a block of 1 token x 1 head x 3 fp16 elements (6 bytes) is not a multiple of 16
    assert lib.paged_kv_swap_blocks(vp(16), vp(16), 4, vp(16), vp(16), 4, vp(16), 2, 1, 1, 3, 1,
                                    None) == INVALID
    assert lib.paged_kv_swap_blocks(vp(16), vp(16), 0, vp(16), vp(16), 4, vp(16), 2, 8, 1, 8, 1,
                                    None) == INVALID
    assert lib.paged_kv_swap_blocks(vp(16), vp(16), 4, vp(16), vp(16), 4, vp(16), -1, 8, 1, 8, 1,
                                    None) == INVALID
    assert lib.paged_kv_swap_blocks(vp(16), vp(16), 4, vp(16), vp(16), 4, vp(16), 2, 8, 1, 8, 7,
                                    None) == INVALID
    assert lib.paged_kv_swap_blocks(vp(0), vp(0), 4, vp(0), vp(0), 4, vp(0), 0, 8, 1, 8, 1,
                                    None) == 0
    # a pool the device cannot reach (no device here at all, or pageable memory)
    buf = (ctypes.c_uint8 * 4096)()
    a = ctypes.cast(buf, vp)
    assert lib.paged_kv_swap_blocks(a, a, 4, a, a, 4, a, 1, 8, 1, 8, 1, None) == INVALID
    assert lib.paged_kv_copy_blocks(vp(16), vp(16), vp(16), 1, 4, 1, 1, 3, 1, None) == INVALID
    assert lib.paged_kv_copy_blocks(vp(0), vp(0), vp(0), 0, 4, 8, 1, 8, 1, None) == 0


def test_workspace_size_follows_the_documented_layout(lib):
    def r256(x):
        return (x + 255) // 256 * 256
    for S, Hq, D, MB, B, P in [(8, 64, 128, 8192, 16, 512), (4, 4, 64, 5, 16, 16), (3, 2, 64, 7, 8, 48)]:
        parts = -(-(MB * B) // P)
        rows = S * Hq * parts
        want = r256(rows * D * 4) + 2 * r256(rows * 4)
        assert pk.paged_attention_workspace_bytes(S, Hq, D, MB, B, P) == want
    assert pk.paged_attention_workspace_bytes(8, 64, 128, 100, 16, 0) == 0


def test_options_round_trip(lib):
    old = pk.get_option(pk.OPT_MMA_MIN_GROUP)
    pk.set_option(pk.OPT_MMA_MIN_GROUP, 2)
    assert pk.get_option(pk.OPT_MMA_MIN_GROUP) == 2
    pk.set_option(pk.OPT_MMA_MIN_GROUP, old)
    with pytest.raises(pk.PagedKVError):
        pk.set_option(pk.OPT_DECODE_PATH, 9)
    with pytest.raises(pk.PagedKVError):
        pk.set_option(99, 0)
    with pytest.raises(pk.PagedKVError):
        pk.set_option(pk.OPT_STAGES, 1)
    pk.set_option(pk.OPT_STAGES, 3)
    assert pk.get_option(pk.OPT_STAGES) == 3
    pk.set_option(pk.OPT_STAGES, 0)
    assert pk.get_option(pk.OPT_L2_HINTS) == 0          # automatic by default
    for mode in (1, 2, 0):
        pk.set_option(pk.OPT_L2_HINTS, mode)
        assert pk.get_option(pk.OPT_L2_HINTS) == mode
    with pytest.raises(pk.PagedKVError):
        pk.set_option(pk.OPT_L2_HINTS, 3)


def test_tensors_must_be_on_the_gpu(lib):
    import torch
    h = torch.zeros(8, 16, 2, 64)     # pageable host memory: the swap refuses it too
    with pytest.raises(pk.PagedKVError, match="pinned"):
        pk.paged_kv_swap_blocks(h, h, h, h, torch.zeros(1, 2, dtype=torch.int32))
    x = torch.zeros(4, 2, 64)
    with pytest.raises(pk.PagedKVError, match="CUDA"):
        pk.paged_kv_append(x, x, torch.zeros(4, dtype=torch.int64), torch.zeros(8, 16, 2, 64),
                           torch.zeros(8, 16, 2, 64))


def test_prefill_key_split_host_checks(lib):
    """The key split's part count is checked before anything reaches the
    device, and its workspace size is plain arithmetic: fp32 outputs
    [parts][tokens * heads][head_dim], then m and l [parts][tokens * heads],
    each rounded up to 256 bytes."""
    vp = ctypes.c_void_p

    def call(parts):
        return lib.paged_attention_prefill_split(vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), 0.1,
                                                 vp(16), 2, 64, 32, 32, 32, 128, 64, 16, 8, 1, parts,
                                                 None, 0, None)

    assert call(33) == INVALID
    assert call(-1) == INVALID
    # the split's workspace depends on the device's SM count: none without a device
    for d in (32, 64, 96, 128):
        assert lib.paged_attention_prefill_workspace_bytes(d) == 0
