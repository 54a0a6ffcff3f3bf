"""GB300-native paged KV cache: append and fused paged-attention decode.

A thin ctypes binding over ``libpagedkv.so`` (C ABI in ``include/pagedkv.h``).
It only marshals torch tensors into pointers and sizes: every step of the
path runs in the library's CUDA kernels, and there is no CPU fallback. If the
library has not been built, the first call raises ``PagedKVError`` (build it
with ``python -m paged_kv_cache_233_gb300.build``).

The entry points keep the C names:

    paged_kv_slot_mapping(block_tables, token_seq, token_pos, slot_mapping, num_blocks, block_size)
    paged_kv_append(k, v, slot_mapping, k_cache, v_cache)
    paged_kv_append_tokens(k, v, block_tables, token_seq, token_pos, k_cache, v_cache,
                           slot_mapping=None)
    paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                           partition_tokens=0, workspace=None)
    paged_attention_workspace_bytes(num_seqs, n_q_heads, head_dim, max_blocks_per_seq,
                                    block_size, partition_tokens)

All tensors live on the current CUDA device; work is enqueued on the current
torch stream (or the stream passed) and the calls return without waiting.
"""
import ctypes
import os

import torch

__all__ = [
    "PagedKVError", "paged_kv_slot_mapping", "paged_kv_append", "paged_attention_decode",
    "paged_attention_workspace_bytes", "new_workspace", "device_errors", "set_option",
    "get_option", "last_decode_path", "status_string", "abi_version", "library_path", "load",
    "DTYPE_CODES", "OPT_DECODE_PATH", "OPT_CTAS_PER_SM", "OPT_MMA_MIN_GROUP", "OPT_STAGES",
    "OPT_PREFILL_PATH", "OPT_L2_HINTS",
    "paged_attention_decode_noalloc", "NOALLOC_SCRATCH_BYTES", "PARTITION_BALANCED",
    "paged_kv_copy_blocks", "paged_attention_decode_shared_prefix", "paged_kv_swap_blocks",
    "paged_attention_prefill", "paged_kv_append_tokens", "check_bounded_wait", "DEVERR_TIMEOUT",
    "prefill_workspace_bytes", "prefill_workspace",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

DTYPE_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
OPT_DECODE_PATH, OPT_CTAS_PER_SM, OPT_MMA_MIN_GROUP, OPT_STAGES, OPT_PREFILL_PATH = 1, 2, 3, 4, 5
OPT_L2_HINTS = 6
NOALLOC_SCRATCH_BYTES = 64 << 20   # PAGEDKV_NOALLOC_SCRATCH_BYTES
PARTITION_BALANCED = -1            # PAGEDKV_PARTITION_BALANCED
DEVERR_TIMEOUT = 0x20              # PAGEDKV_DEVERR_TIMEOUT: a bounded in-kernel wait gave up
EXPORTS = ("paged_kv_slot_mapping", "paged_kv_append", "paged_attention_decode",
           "paged_attention_workspace_bytes", "pagedkv_device_errors", "pagedkv_set_option",
           "pagedkv_get_option", "pagedkv_last_decode_path", "pagedkv_status_string",
           "pagedkv_abi_version", "paged_attention_decode_noalloc", "paged_kv_copy_blocks",
           "paged_attention_decode_shared_prefix", "paged_kv_append_tokens",
           "pagedkv_check_bounded_wait", "paged_attention_prefill_split",
           "paged_attention_prefill_workspace_bytes")


class PagedKVError(RuntimeError):
    pass


_lib = None


def library_path():
    return _LIB_PATH


def load():
    """Load libpagedkv.so (once). Raises PagedKVError when it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise PagedKVError(
            f"{_LIB_PATH} is not built: run `python -m paged_kv_cache_233_gb300.build` "
            "(the paged-KV path has no fallback)")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.paged_kv_slot_mapping.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
    lib.paged_kv_append.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]
    lib.paged_kv_append_tokens.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                           i32, i32, i32, vp]
    lib.paged_kv_append_tokens.restype = i32
    lib.paged_attention_decode.argtypes = [vp, vp, vp, vp, vp, ctypes.c_float, vp, i32, i32, i32,
                                           i32, i32, i32, i32, i32, vp, sz, i32, vp]
    lib.paged_attention_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, ctypes.c_float, vp, i32,
                                                   i32, i32, i32, i32, i32, i32, i32, i32, vp]
    lib.paged_attention_decode_noalloc.restype = i32
    lib.paged_attention_decode_shared_prefix.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32,
                                                         ctypes.c_float, vp, i32, i32, i32, i32,
                                                         i32, i32, i32, i32, vp, sz, i32, vp]
    lib.paged_attention_decode_shared_prefix.restype = i32
    lib.paged_kv_copy_blocks.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]
    lib.paged_kv_copy_blocks.restype = i32
    lib.paged_kv_swap_blocks.argtypes = [vp, vp, i32, vp, vp, i32, vp, i32, i32, i32, i32, i32, vp]
    lib.paged_kv_swap_blocks.restype = i32
    lib.paged_attention_prefill.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, i32, i32,
                                            i32, i32, i32, i32, i32, i32, i32, i32, vp]
    lib.paged_attention_prefill.restype = i32
    lib.paged_attention_prefill_split.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, i32,
                                                  i32, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                                  vp, sz, vp]
    lib.paged_attention_prefill_split.restype = i32
    lib.paged_attention_prefill_workspace_bytes.argtypes = [i32]
    lib.paged_attention_prefill_workspace_bytes.restype = sz
    lib.paged_attention_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.paged_attention_workspace_bytes.restype = sz
    lib.pagedkv_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint), i32]
    lib.pagedkv_check_bounded_wait.argtypes = [vp]
    lib.pagedkv_check_bounded_wait.restype = i32
    lib.pagedkv_set_option.argtypes = [i32, i32]
    lib.pagedkv_get_option.argtypes = [i32]
    lib.pagedkv_status_string.argtypes = [i32]
    lib.pagedkv_status_string.restype = ctypes.c_char_p
    for name in ("paged_kv_slot_mapping", "paged_kv_append", "paged_attention_decode",
                 "pagedkv_device_errors", "pagedkv_set_option", "pagedkv_get_option",
                 "pagedkv_last_decode_path", "pagedkv_abi_version"):
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


def status_string(status):
    return load().pagedkv_status_string(int(status)).decode()


def abi_version():
    return load().pagedkv_abi_version()


def _check(status, what):
    if status != 0:
        raise PagedKVError(f"{what}: {status_string(status)} ({status})")


# The current stream's raw handle without building a torch Stream object
# (about 0.1 us instead of 3 us per call); torch.cuda.current_stream() where
# this torch lacks the accessor.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    """The CUDA stream handle (an int; 0 is the legacy default stream)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _dev(t, name, dtype=None):
    """The device address of a contiguous CUDA tensor (an int), checked."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise PagedKVError(f"{name} must be a CUDA tensor (the paged-KV path has no CPU fallback)")
    if not t.is_contiguous():
        raise PagedKVError(f"{name} must be contiguous")
    if dtype is not None and t.dtype is not dtype:
        raise PagedKVError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _code(t):
    try:
        return DTYPE_CODES[t.dtype]
    except KeyError:
        raise PagedKVError(f"unsupported element type {t.dtype}") from None


def paged_kv_slot_mapping(block_tables, token_seq, token_pos, slot_mapping, num_blocks, block_size,
                          stream=None):
    """slot_mapping[t] = block_tables[seq][pos // B] * B + pos % B (int64; -1 for padding)."""
    n = token_seq.numel()
    if token_pos.numel() != n or slot_mapping.numel() != n:
        raise PagedKVError("token_seq, token_pos and slot_mapping differ in length")
    st = load().paged_kv_slot_mapping(
        _dev(block_tables, "block_tables", torch.int32), _dev(token_seq, "token_seq", torch.int32),
        _dev(token_pos, "token_pos", torch.int32), _dev(slot_mapping, "slot_mapping", torch.int64),
        n, block_tables.shape[0], block_tables.shape[1], int(block_size), int(num_blocks),
        _stream(stream))
    _check(st, "paged_kv_slot_mapping")


def paged_kv_append(k, v, slot_mapping, k_cache, v_cache, stream=None):
    """Scatter k/v [T][Hkv][D] into the pools [NB][B][Hkv][D] at slot_mapping[T]."""
    ks, cs = k.shape, k_cache.shape
    if len(ks) != 3 or v.shape != ks or len(cs) != 4 or v_cache.shape != cs:
        raise PagedKVError("expected k, v [T][Hkv][D] and pools [NB][B][Hkv][D]")
    if not (k.dtype is v.dtype is k_cache.dtype is v_cache.dtype):
        raise PagedKVError("k, v and the pools must share one element type")
    NB, B, Hkv, D = cs
    T = ks[0]
    if ks[1] != Hkv or ks[2] != D:
        raise PagedKVError("token rows do not match the pool's [Hkv][D]")
    if slot_mapping.numel() != T:
        raise PagedKVError("slot_mapping length differs from the number of tokens")
    st = load().paged_kv_append(
        _dev(k, "k"), _dev(v, "v"), _dev(slot_mapping, "slot_mapping", torch.int64),
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), T, NB, B, Hkv, D, _code(k),
        _stream(stream))
    _check(st, "paged_kv_append")


def paged_kv_append_tokens(k, v, block_tables, token_seq, token_pos, k_cache, v_cache,
                           slot_mapping=None, stream=None):
    """paged_kv_slot_mapping and paged_kv_append in one launch: token t's K/V
    rows go to slot block_tables[seq][pos // B] * B + pos % B (seq, pos =
    token_seq[t], token_pos[t]; negative pos is padding); the slots are also
    written to slot_mapping (int64) when it is given."""
    ks, cs = k.shape, k_cache.shape
    if len(ks) != 3 or v.shape != ks or len(cs) != 4 or v_cache.shape != cs:
        raise PagedKVError("expected k, v [T][Hkv][D] and pools [NB][B][Hkv][D]")
    if not (k.dtype is v.dtype is k_cache.dtype is v_cache.dtype):
        raise PagedKVError("k, v and the pools must share one element type")
    NB, B, Hkv, D = cs
    T = ks[0]
    if ks[1] != Hkv or ks[2] != D:
        raise PagedKVError("token rows do not match the pool's [Hkv][D]")
    if token_seq.numel() != T or token_pos.numel() != T or block_tables.dim() != 2:
        raise PagedKVError("token_seq and token_pos need one entry per token, block_tables 2 dims")
    sm = None
    if slot_mapping is not None:
        if slot_mapping.numel() != T:
            raise PagedKVError("slot_mapping length differs from the number of tokens")
        sm = _dev(slot_mapping, "slot_mapping", torch.int64)
    st = load().paged_kv_append_tokens(
        _dev(k, "k"), _dev(v, "v"), _dev(block_tables, "block_tables", torch.int32),
        _dev(token_seq, "token_seq", torch.int32), _dev(token_pos, "token_pos", torch.int32), sm,
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), T, block_tables.shape[0],
        block_tables.shape[1], NB, B, Hkv, D, _code(k), _stream(stream))
    _check(st, "paged_kv_append_tokens")


def paged_kv_copy_blocks(k_cache, v_cache, block_pairs, stream=None):
    """Copy-on-write: copy whole blocks block_pairs[i][0] -> block_pairs[i][1] in both pools."""
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise PagedKVError("expected pools [NB][B][Hkv][D] of one element type")
    if block_pairs.dim() != 2 or block_pairs.shape[1] != 2:
        raise PagedKVError("block_pairs must be [n][2]")
    NB, B, Hkv, D = k_cache.shape
    st = load().paged_kv_copy_blocks(
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_pairs, "block_pairs", torch.int32), block_pairs.shape[0], NB, B, Hkv, D,
        _code(k_cache), _stream(stream))
    _check(st, "paged_kv_copy_blocks")


def _reachable(t, name, dtype=None):
    """A tensor the GPU can address in place: CUDA memory or pinned host memory."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_contiguous():
        raise PagedKVError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise PagedKVError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda and not t.is_pinned():
        raise PagedKVError(f"{name} must be a CUDA tensor or pinned host memory")
    return t.data_ptr()


def paged_kv_swap_blocks(src_k, src_v, dst_k, dst_v, block_pairs, stream=None):
    """Copy whole blocks block_pairs[i][0] of the source pools to block_pairs[i][1]
    of the destination pools (swap-out to pinned host pools, or swap-in back).

    Pools are [NB][B][Hkv][D] of one element type; source and destination may
    hold different numbers of blocks. Any argument may live in CUDA memory or in
    pinned host memory; the copy runs on the GPU, asynchronously on `stream`.
    """
    for a, b, what in ((src_k, src_v, "source"), (dst_k, dst_v, "destination")):
        if a.dim() != 4 or a.shape != b.shape or a.dtype != b.dtype:
            raise PagedKVError(f"expected {what} pools [NB][B][Hkv][D] of one element type")
    if src_k.shape[1:] != dst_k.shape[1:] or src_k.dtype != dst_k.dtype:
        raise PagedKVError("source and destination blocks differ in shape or element type")
    if block_pairs.dim() != 2 or block_pairs.shape[1] != 2:
        raise PagedKVError("block_pairs must be [n][2]")
    _, B, Hkv, D = src_k.shape
    st = load().paged_kv_swap_blocks(
        _reachable(src_k, "src_k"), _reachable(src_v, "src_v"), src_k.shape[0],
        _reachable(dst_k, "dst_k"), _reachable(dst_v, "dst_v"), dst_k.shape[0],
        _reachable(block_pairs, "block_pairs", torch.int32), block_pairs.shape[0], B, Hkv, D,
        _code(src_k), _stream(stream))
    _check(st, "paged_kv_swap_blocks")


def paged_attention_prefill(q, k_cache, v_cache, block_tables, query_start, context_lens, scale,
                            out, max_query_len=None, stream=None, workspace=None, key_parts=1):
    """Chunked-prefill attention: q/out [num_tokens][Hq][D] hold every sequence's
    chunk of query rows, sequence after sequence, delimited by query_start
    [num_seqs + 1]; context_lens counts each sequence's cached tokens with its
    chunk (already appended) included. max_query_len bounds every chunk's
    length; by default it is read from query_start (a device-to-host copy).
    With key_parts other than 1 the call's key tiles may be shared out in
    equal ranges over the SMs, no item in more than key_parts of them (0: when
    the items leave SMs idle and the workspace holds the split), and a merge
    kernel combines the pieces' states; the workspace (see prefill_workspace)
    is taken from torch's allocator when none is given."""
    if q.dim() != 3 or out.shape != q.shape or out.dtype != q.dtype:
        raise PagedKVError("q and out must be [num_tokens][n_q_heads][head_dim] of one type")
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape or k_cache.dtype != q.dtype:
        raise PagedKVError("expected pools [NB][B][Hkv][D] of q's element type")
    S = context_lens.shape[0]
    if query_start.shape[0] != S + 1 or block_tables.shape[0] != S:
        raise PagedKVError("query_start must hold num_seqs + 1 offsets, block_tables num_seqs rows")
    if max_query_len is None:
        max_query_len = int((query_start[1:] - query_start[:-1]).max().item()) if S else 0
    NB, B, Hkv, D = k_cache.shape
    args = (_dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
            _dev(block_tables, "block_tables", torch.int32), _dev(query_start, "query_start", torch.int32),
            _dev(context_lens, "context_lens", torch.int32), float(scale), _dev(out, "out"), S,
            q.shape[0], int(max_query_len), q.shape[1], Hkv, D, NB, B, block_tables.shape[1], _code(q))
    if workspace is None and key_parts == 1:
        st = load().paged_attention_prefill(*args, _stream(stream))
        _check(st, "paged_attention_prefill")
        return
    if workspace is None:
        workspace = prefill_workspace(q)
    ws = _dev(workspace, "workspace")
    nbytes = workspace.numel() * workspace.element_size()
    st = load().paged_attention_prefill_split(*args, int(key_parts), ws, nbytes, _stream(stream))
    _check(st, "paged_attention_prefill_split")


def prefill_workspace_bytes(head_dim):
    """Workspace bytes of a prefill whose keys are split, on the current device
    (it depends on the SM count alone; 0 without a device)."""
    return load().paged_attention_prefill_workspace_bytes(int(head_dim))


def prefill_workspace(q):
    """A device buffer for paged_attention_prefill(..., workspace=..., key_parts=...)
    on q's device."""
    with torch.cuda.device(q.device):
        n = prefill_workspace_bytes(q.shape[2])
    return torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)


def paged_attention_workspace_bytes(num_seqs, n_q_heads, head_dim, max_blocks_per_seq, block_size,
                                    partition_tokens):
    return load().paged_attention_workspace_bytes(int(num_seqs), int(n_q_heads), int(head_dim),
                                                  int(max_blocks_per_seq), int(block_size),
                                                  int(partition_tokens))


def new_workspace(q, block_tables, block_size, partition_tokens):
    """A device buffer large enough for split-K decode with these shapes (None if not split)."""
    n = paged_attention_workspace_bytes(q.shape[0], q.shape[1], q.shape[2], block_tables.shape[1],
                                        block_size, partition_tokens)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def _decode_shapes(q, k_cache, v_cache, block_tables, context_lens, out):
    """(S, Hq, Hkv, D, NB, B, max_blocks) of a decode call, checked."""
    qs, cs, bs = q.shape, k_cache.shape, block_tables.shape
    if len(qs) != 3 or out.shape != qs or len(cs) != 4 or v_cache.shape != cs:
        raise PagedKVError("expected q/out [S][Hq][D] and pools [NB][B][Hkv][D]")
    if not (q.dtype is out.dtype is k_cache.dtype is v_cache.dtype):
        raise PagedKVError("q, out and the pools must share one element type")
    S, Hq, D = qs
    NB, B, Hkv, Dk = cs
    if Dk != D or len(bs) != 2 or bs[0] != S or context_lens.numel() != S:
        raise PagedKVError("shape mismatch between q, the pools, block_tables and context_lens")
    return S, Hq, Hkv, D, NB, B, bs[1]


def paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                           partition_tokens=0, workspace=None, stream=None):
    """out[s][h] = softmax(scale * q[s][h] . K_s) V_s with K_s, V_s read through block_tables.

    partition_tokens: 0 = no split, > 0 = split-K in partitions of that many
    tokens, PARTITION_BALANCED = equal tile shares per CTA; splits need a
    workspace (new_workspace)."""
    S, Hq, Hkv, D, NB, B, MB = _decode_shapes(q, k_cache, v_cache, block_tables, context_lens, out)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    st = load().paged_attention_decode(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32),
        _dev(context_lens, "context_lens", torch.int32), float(scale), _dev(out, "out"), S, Hq, Hkv,
        D, NB, B, MB, int(partition_tokens), ws_ptr, ws_bytes, _code(q), _stream(stream))
    _check(st, "paged_attention_decode")


def paged_attention_decode_shared_prefix(q, k_cache, v_cache, block_tables, context_lens, seq_group,
                                         group_prefix, scale, out, partition_tokens, workspace,
                                         stream=None):
    """paged_attention_decode for batches whose consecutive sequences share
    prefixes: seq_group[s] (int32, -1 = none) names each sequence's group and
    group_prefix[g] (int32) the tokens every member holds in the group's first
    member's blocks. Each shared prefix partition is read once per chunk of
    members instead of once per member. Needs a split (partition_tokens > 0)."""
    S, Hq, Hkv, D, NB, B, MB = _decode_shapes(q, k_cache, v_cache, block_tables, context_lens, out)
    if seq_group.numel() != S:
        raise PagedKVError("shape mismatch between q, the pools, block_tables, lengths and groups")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    st = load().paged_attention_decode_shared_prefix(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32),
        _dev(context_lens, "context_lens", torch.int32), _dev(seq_group, "seq_group", torch.int32),
        _dev(group_prefix, "group_prefix", torch.int32), group_prefix.numel(), float(scale),
        _dev(out, "out"), S, Hq, Hkv, D, NB, B, MB, int(partition_tokens), ws_ptr, ws_bytes,
        _code(q), _stream(stream))
    _check(st, "paged_attention_decode_shared_prefix")


def paged_attention_decode_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                                   partition_tokens=0, stream=None):
    """paged_attention_decode without a workspace argument, for callers that must
    not allocate device memory on their call path (a serving loop with a fixed
    latency budget, a plug-in whose host owns all device memory, a process whose
    free memory belongs to another allocator). Split-K partition states go to a
    fixed library-owned device array of NOALLOC_SCRATCH_BYTES shared by every
    call on the device: order such calls on one stream. A split that needs more
    than that raises PagedKVError (status -5)."""
    S, Hq, Hkv, D, NB, B, MB = _decode_shapes(q, k_cache, v_cache, block_tables, context_lens, out)
    st = load().paged_attention_decode_noalloc(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32),
        _dev(context_lens, "context_lens", torch.int32), float(scale), _dev(out, "out"), S, Hq, Hkv,
        D, NB, B, MB, int(partition_tokens), _code(q), _stream(stream))
    _check(st, "paged_attention_decode_noalloc")


def check_bounded_wait(stream=None):
    """Enqueue a kernel whose bounded wait on a barrier that nothing arrives on
    gives up (after 1 s) and sets the timeout bit of device_errors()."""
    _check(load().pagedkv_check_bounded_wait(_stream(stream)), "pagedkv_check_bounded_wait")


def device_errors(reset=True):
    """The sticky device error bits (synchronises the device); 0 when clean."""
    flags = ctypes.c_uint(0)
    st = load().pagedkv_device_errors(ctypes.byref(flags), 1 if reset else 0)
    if st not in (0, -4):
        _check(st, "pagedkv_device_errors")
    return flags.value


def set_option(option, value):
    _check(load().pagedkv_set_option(int(option), int(value)), "pagedkv_set_option")


def get_option(option):
    return load().pagedkv_get_option(int(option))


def last_decode_path():
    return load().pagedkv_last_decode_path()
