"""fp64 CPU oracle for paged KV append and paged-attention decode.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by ``bench.py``'s CPU-baseline leg, never by the product package. It
shares no code with the CUDA library. The arithmetic lives in
``pagedkv_oracle.c``; this module only marshals numpy arrays into it.

Element type names: "f32", "f16", "bf16". Arrays of 16-bit types may be
passed as float16 or as raw uint16/int16 bit patterns; they are read as
bits either way.

Every function is pinned in ``tests/test_oracle_pins.py`` against something
other than itself: numpy's own contiguous softmax attention, invariances of
the definition, closed-form special cases and the pages' worked examples.
"""
import ctypes
import os

import numpy as np

from . import build as _build

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}
ELEMENT_BYTES = {"f32": 4, "f16": 2, "bf16": 2}

_c_i32p = ctypes.POINTER(ctypes.c_int32)
_c_i64p = ctypes.POINTER(ctypes.c_int64)
_c_f64p = ctypes.POINTER(ctypes.c_double)
_c_u8p = ctypes.POINTER(ctypes.c_uint8)


def _ptr(a, ctype=ctypes.c_void_p):
    return ctypes.cast(a.ctypes.data, ctype)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _raw(a, dtype):
    """The array's bytes, checked against the element type's size."""
    a = np.ascontiguousarray(a)
    if a.dtype.itemsize != ELEMENT_BYTES[dtype]:
        raise TypeError(f"array of {a.dtype} does not hold {dtype} elements")
    return a


class Oracle:
    """Bindings to one build of the oracle library."""

    def __init__(self, path=None):
        self.path = path or _build.build()
        lib = ctypes.CDLL(self.path)
        lib.oracle_f16_to_double.restype = ctypes.c_double
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_slot.restype = ctypes.c_int64
        lib.oracle_slot.argtypes = [_c_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                    ctypes.c_int]
        lib.oracle_slot_mapping.restype = ctypes.c_int
        lib.oracle_slot_mapping.argtypes = [_c_i32p, ctypes.c_int, _c_i32p, _c_i32p,
                                            ctypes.c_int64, ctypes.c_int, _c_i64p]
        lib.oracle_append.restype = ctypes.c_int64
        lib.oracle_append.argtypes = [_c_u8p, _c_u8p, _c_i64p, ctypes.c_int64, _c_u8p, _c_u8p,
                                      ctypes.c_int64, ctypes.c_int64]
        lib.oracle_copy_blocks.restype = ctypes.c_int64
        lib.oracle_copy_blocks.argtypes = [_c_u8p, _c_u8p, _c_i32p, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int64]
        lib.oracle_swap_blocks.restype = ctypes.c_int64
        lib.oracle_swap_blocks.argtypes = [_c_u8p, _c_u8p, ctypes.c_int64, _c_u8p, _c_u8p,
                                           ctypes.c_int64, _c_i32p, ctypes.c_int64,
                                           ctypes.c_int64]
        lib.oracle_gather.restype = None
        lib.oracle_gather.argtypes = [ctypes.c_void_p, _c_i32p, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, _c_f64p]
        lib.oracle_decode_units.restype = ctypes.c_int
        lib.oracle_decode_units.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, _c_i32p, _c_i32p,
            ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_i32p, ctypes.c_int64, _c_f64p,
            ctypes.c_int]
        lib.oracle_prefill_units.restype = ctypes.c_int
        lib.oracle_prefill_units.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, _c_i32p, _c_i32p, _c_i32p,
            ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, _c_i32p, ctypes.c_int64, _c_f64p, ctypes.c_int]
        lib.oracle_decode_partition.restype = ctypes.c_int
        lib.oracle_decode_partition.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, _c_i32p, ctypes.c_double,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_f64p, _c_f64p, _c_f64p]
        lib.oracle_lse_merge.restype = None
        lib.oracle_lse_merge.argtypes = [ctypes.c_int, _c_f64p, _c_f64p, _c_f64p, ctypes.c_int,
                                         _c_f64p]
        lib.oracle_max_threads.restype = ctypes.c_int
        self.lib = lib

    # -- element decoding ---------------------------------------------------
    def f16_to_double(self, bits):
        return self.lib.oracle_f16_to_double(int(bits))

    def bf16_to_double(self, bits):
        return self.lib.oracle_bf16_to_double(int(bits))

    def widen(self, a, dtype):
        """All elements of `a` (stored as `dtype`) widened to float64."""
        a = _raw(a, dtype)
        if dtype == "f32":
            return a.view(np.float32).astype(np.float64)
        f = self.f16_to_double if dtype == "f16" else self.bf16_to_double
        flat = a.view(np.uint16).ravel()
        return np.array([f(b) for b in flat], dtype=np.float64).reshape(a.shape)

    # -- address translation --------------------------------------------------
    def slot(self, block_tables, seq, pos, block_size):
        bt = _i32(block_tables)
        return self.lib.oracle_slot(_ptr(bt, _c_i32p), bt.shape[1], int(seq), int(pos),
                                    int(block_size))

    def slot_mapping(self, block_tables, token_seq, token_pos, block_size):
        """slot_mapping[t] for tokens (token_seq[t], token_pos[t]); -1 for padding."""
        bt, ts, tp = _i32(block_tables), _i32(token_seq), _i32(token_pos)
        out = np.empty(ts.shape[0], dtype=np.int64)
        st = self.lib.oracle_slot_mapping(_ptr(bt, _c_i32p), bt.shape[1], _ptr(ts, _c_i32p),
                                          _ptr(tp, _c_i32p), ts.shape[0], int(block_size),
                                          _ptr(out, _c_i64p))
        if st != 0:
            raise IndexError("a token position lies outside its block table")
        return out

    # -- append -----------------------------------------------------------------
    def append(self, k, v, slot_mapping, k_cache, v_cache):
        """Store k[t], v[t] at slot_mapping[t] of the pools, in place.

        k, v: [T][n_kv_heads][head_dim]; pools: [num_blocks][block_size][n_kv_heads][head_dim],
        all of one element type. Returns the number of out-of-range slots skipped.
        """
        k = np.ascontiguousarray(k)
        v = np.ascontiguousarray(v)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        for c in (k_cache, v_cache):
            if not c.flags.c_contiguous:
                raise ValueError("pools must be contiguous")
        row_bytes = k.dtype.itemsize * int(np.prod(k.shape[1:]))
        num_slots = k_cache.shape[0] * k_cache.shape[1]
        if k_cache.dtype.itemsize * int(np.prod(k_cache.shape[2:])) != row_bytes:
            raise ValueError("token rows and pool rows differ in size")
        return self.lib.oracle_append(_ptr(k, _c_u8p), _ptr(v, _c_u8p), _ptr(sm, _c_i64p),
                                      sm.shape[0], _ptr(k_cache, _c_u8p), _ptr(v_cache, _c_u8p),
                                      num_slots, row_bytes)

    # -- copy-on-write ------------------------------------------------------------
    def copy_blocks(self, k_cache, v_cache, pairs):
        """Copy whole blocks src -> dst (pairs [n][2]) in both pools, in place, in order.
        Returns the number of pairs skipped for ids outside the pool."""
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        for c in (k_cache, v_cache):
            if not c.flags.c_contiguous:
                raise ValueError("pools must be contiguous")
        block_bytes = k_cache.dtype.itemsize * int(np.prod(k_cache.shape[1:]))
        return self.lib.oracle_copy_blocks(_ptr(k_cache, _c_u8p), _ptr(v_cache, _c_u8p),
                                           _ptr(pr, _c_i32p), pr.shape[0], k_cache.shape[0],
                                           block_bytes)

    # -- swap between pools ---------------------------------------------------------
    def swap_blocks(self, src_k, src_v, dst_k, dst_v, pairs):
        """Copy whole blocks from the source pools into the destination pools
        (pairs [n][2] = (source block, destination block)), in order, in place.
        Returns the number of pairs skipped for ids outside their pool."""
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        for c in (src_k, src_v, dst_k, dst_v):
            if not c.flags.c_contiguous:
                raise ValueError("pools must be contiguous")
        block_bytes = src_k.dtype.itemsize * int(np.prod(src_k.shape[1:]))
        if dst_k.dtype.itemsize * int(np.prod(dst_k.shape[1:])) != block_bytes:
            raise ValueError("source and destination blocks differ in size")
        return self.lib.oracle_swap_blocks(_ptr(src_k, _c_u8p), _ptr(src_v, _c_u8p),
                                           src_k.shape[0], _ptr(dst_k, _c_u8p),
                                           _ptr(dst_v, _c_u8p), dst_k.shape[0],
                                           _ptr(pr, _c_i32p), pr.shape[0], block_bytes)

    # -- gather -------------------------------------------------------------------
    def gather(self, cache, block_tables, seq, length, kv_head, dtype):
        """[length][head_dim] float64 copy of one sequence's cache for one kv head."""
        cache = _raw(cache, dtype)
        bt = _i32(block_tables)
        _, block_size, n_kv_heads, head_dim = cache.shape
        out = np.empty((max(int(length), 0), head_dim), dtype=np.float64)
        self.lib.oracle_gather(_ptr(cache), _ptr(bt, _c_i32p), bt.shape[1], int(seq),
                               int(length), int(kv_head), n_kv_heads, head_dim, block_size,
                               DTYPE_CODES[dtype], _ptr(out, _c_f64p))
        return out

    # -- decode -------------------------------------------------------------------
    def decode(self, q, k_cache, v_cache, block_tables, context_lens, scale, dtype,
               units=None, threads=0):
        """Decode attention; returns float64 [num_seqs][n_q_heads][head_dim].

        units: optional iterable of (seq, kv_head) pairs to compute; rows of
        other units are NaN. Default: every unit.
        """
        q, k_cache, v_cache = (_raw(x, dtype) for x in (q, k_cache, v_cache))
        bt, lens = _i32(block_tables), _i32(context_lens)
        num_seqs, n_q_heads, head_dim = q.shape
        _, block_size, n_kv_heads, hd = k_cache.shape
        if hd != head_dim or v_cache.shape != k_cache.shape:
            raise ValueError("shape mismatch between q and the pools")
        if units is None:
            units = [(s, h) for s in range(num_seqs) for h in range(n_kv_heads)]
        u = _i32(np.asarray(list(units), dtype=np.int32).reshape(-1, 2))
        out = np.full((num_seqs, n_q_heads, head_dim), np.nan, dtype=np.float64)
        st = self.lib.oracle_decode_units(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt, _c_i32p), _ptr(lens, _c_i32p),
            float(scale), num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, bt.shape[1],
            DTYPE_CODES[dtype], _ptr(u, _c_i32p), u.shape[0], _ptr(out, _c_f64p), int(threads))
        if st != 0:
            raise ValueError("a context length lies outside its block table")
        return out

    def prefill(self, q, k_cache, v_cache, block_tables, query_start, context_lens, scale,
                dtype, units=None, threads=0):
        """Chunked-prefill attention; returns float64 [num_tokens][n_q_heads][head_dim].

        q holds every sequence's chunk of query rows, sequence after sequence;
        query_start[num_seqs + 1] delimits them; context_lens counts each
        sequence's cached tokens with its chunk included. units: optional
        (seq, kv_head) pairs to compute; rows of other units are NaN.
        """
        q, k_cache, v_cache = (_raw(x, dtype) for x in (q, k_cache, v_cache))
        bt, qs, lens = _i32(block_tables), _i32(query_start), _i32(context_lens)
        num_tokens, n_q_heads, head_dim = q.shape
        _, block_size, n_kv_heads, hd = k_cache.shape
        num_seqs = lens.shape[0]
        if hd != head_dim or v_cache.shape != k_cache.shape:
            raise ValueError("shape mismatch between q and the pools")
        if qs.shape[0] != num_seqs + 1 or qs[0] != 0 or qs[-1] != num_tokens or (np.diff(qs) < 0).any():
            raise ValueError("query_start must run from 0 to num_tokens without decreasing")
        if units is None:
            units = [(s, h) for s in range(num_seqs) for h in range(n_kv_heads)]
        u = _i32(np.asarray(list(units), dtype=np.int32).reshape(-1, 2))
        out = np.full((num_tokens, n_q_heads, head_dim), np.nan, dtype=np.float64)
        st = self.lib.oracle_prefill_units(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt, _c_i32p), _ptr(qs, _c_i32p),
            _ptr(lens, _c_i32p), float(scale), n_q_heads, n_kv_heads, head_dim, block_size,
            bt.shape[1], DTYPE_CODES[dtype], _ptr(u, _c_i32p), u.shape[0], _ptr(out, _c_f64p),
            int(threads))
        if st != 0:
            raise ValueError("a chunk is longer than its context, or a context lies outside its table")
        return out

    def decode_partition(self, q, k_cache, v_cache, block_tables, scale, dtype, seq, qh,
                         t0, t1):
        """(o[head_dim], m, l): unnormalised state of head qh over tokens [t0, t1)."""
        q, k_cache, v_cache = (_raw(x, dtype) for x in (q, k_cache, v_cache))
        bt = _i32(block_tables)
        _, n_q_heads, head_dim = q.shape
        _, block_size, n_kv_heads, _ = k_cache.shape
        o = np.empty(head_dim, dtype=np.float64)
        m = np.empty(1, dtype=np.float64)
        l = np.empty(1, dtype=np.float64)
        st = self.lib.oracle_decode_partition(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt, _c_i32p), float(scale), n_q_heads,
            n_kv_heads, head_dim, block_size, bt.shape[1], DTYPE_CODES[dtype], int(seq),
            int(qh), int(t0), int(t1), _ptr(o, _c_f64p), _ptr(m, _c_f64p), _ptr(l, _c_f64p))
        if st != 0:
            raise ValueError("bad partition range")
        return o, float(m[0]), float(l[0])

    def lse_merge(self, m, l, o):
        """Normalised output row from partition states m[n], l[n], o[n][head_dim]."""
        m = np.ascontiguousarray(m, dtype=np.float64)
        l = np.ascontiguousarray(l, dtype=np.float64)
        o = np.ascontiguousarray(o, dtype=np.float64)
        out = np.empty(o.shape[1], dtype=np.float64)
        self.lib.oracle_lse_merge(m.shape[0], _ptr(m, _c_f64p), _ptr(l, _c_f64p),
                                  _ptr(o, _c_f64p), o.shape[1], _ptr(out, _c_f64p))
        return out

    def max_threads(self):
        return self.lib.oracle_max_threads()


_default = None


def get():
    """The oracle built from this directory's source (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def library_path():
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "liboracle.so")
