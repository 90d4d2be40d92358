"""CPU oracle for paged KV-cache attention (ctypes front end of oracle.cpp).

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg use this module; the CUDA library never does.
It shares no code with the CUDA path.  Inputs are numpy arrays; 16-bit floats
travel as their uint16 bit patterns, E4M3 as uint8.

Everything here is a thin marshalling layer over the C++ in oracle.cpp; the
arithmetic and the citations live there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16, BF16, E4M3 = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.cpp into liboracle.so with g++ (-O2, IEEE arithmetic)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_D = ctypes.c_double
_F = ctypes.c_float


def _declare(L):
    L.orc_decode_f16.restype = _D
    L.orc_decode_f16.argtypes = [ctypes.c_uint16]
    L.orc_decode_bf16.restype = _D
    L.orc_decode_bf16.argtypes = [ctypes.c_uint16]
    L.orc_decode_e4m3.restype = _D
    L.orc_decode_e4m3.argtypes = [ctypes.c_uint8]
    L.orc_encode_e4m3.restype = ctypes.c_uint8
    L.orc_encode_e4m3.argtypes = [_F]
    L.orc_decode_array.restype = None
    L.orc_decode_array.argtypes = [_P, _P, _I64, _I]
    L.orc_encode_e4m3_array.restype = None
    L.orc_encode_e4m3_array.argtypes = [_P, _P, _I64]
    L.orc_kv_bytes_per_token.restype = ctypes.c_uint64
    L.orc_kv_bytes_per_token.argtypes = [_I, _I, _I, _I]
    L.orc_blocks_for_tokens.restype = _I64
    L.orc_blocks_for_tokens.argtypes = [_I64, _I]
    L.orc_pool_create.restype = _P
    L.orc_pool_create.argtypes = [_I, _P]
    L.orc_pool_destroy.restype = None
    L.orc_pool_destroy.argtypes = [_P]
    for name in ("orc_pool_alloc", "orc_pool_num_free"):
        getattr(L, name).restype = _I
    L.orc_pool_alloc.argtypes = [_P]
    L.orc_pool_num_free.argtypes = [_P]
    for name in ("orc_pool_incref", "orc_pool_decref", "orc_pool_ref_cnt"):
        getattr(L, name).restype = _I
        getattr(L, name).argtypes = [_P, _I]
    L.orc_seq_create.restype = _P
    L.orc_seq_create.argtypes = [_P, _I]
    L.orc_seq_destroy.restype = None
    L.orc_seq_destroy.argtypes = [_P]
    L.orc_seq_fork.restype = _P
    L.orc_seq_fork.argtypes = [_P]
    L.orc_seq_append.restype = _I
    L.orc_seq_append.argtypes = [_P, _I, _P, _P, _I64, _P]
    L.orc_seq_num_tokens.restype = _I
    L.orc_seq_num_tokens.argtypes = [_P]
    L.orc_seq_num_blocks.restype = _I
    L.orc_seq_num_blocks.argtypes = [_P]
    L.orc_seq_table.restype = _I
    L.orc_seq_table.argtypes = [_P, _P, _I]
    L.orc_seq_slot.restype = _I64
    L.orc_seq_slot.argtypes = [_P, _I]
    L.orc_cpool_create.restype = _P
    L.orc_cpool_create.argtypes = [_I, _I]
    L.orc_cpool_destroy.restype = None
    L.orc_cpool_destroy.argtypes = [_P]
    for name in ("orc_cpool_num_free", "orc_cpool_num_cached"):
        getattr(L, name).restype = _I
        getattr(L, name).argtypes = [_P]
    for name in ("orc_cpool_ref_cnt", "orc_cpool_is_cached"):
        getattr(L, name).restype = _I
        getattr(L, name).argtypes = [_P, _I]
    L.orc_cpool_queue.restype = _I
    L.orc_cpool_queue.argtypes = [_P, _P, _I]
    L.orc_creq_create.restype = _P
    L.orc_creq_create.argtypes = [_P]
    L.orc_creq_match.restype = _I
    L.orc_creq_match.argtypes = [_P, _P, _I]
    L.orc_creq_append.restype = _I
    L.orc_creq_append.argtypes = [_P, _P, _I, _P, _P]
    L.orc_creq_fork.restype = _P
    L.orc_creq_fork.argtypes = [_P]
    L.orc_creq_free.restype = None
    L.orc_creq_free.argtypes = [_P]
    L.orc_creq_num_tokens.restype = _I
    L.orc_creq_num_tokens.argtypes = [_P]
    L.orc_creq_table.restype = _I
    L.orc_creq_table.argtypes = [_P, _P, _I]
    L.orc_copy_blocks.restype = _I
    L.orc_copy_blocks.argtypes = [_P, _P, _P, _I, _I, _I64]
    L.orc_reshape_and_cache.restype = _I
    L.orc_reshape_and_cache.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _F]
    L.orc_paged_attention_decode.restype = _I
    L.orc_paged_attention_decode.argtypes = [_P] * 6 + [_I] * 7 + [_D, _I, _I, _D, _D]
    L.orc_paged_attention_decode_partitioned.restype = _I
    L.orc_paged_attention_decode_partitioned.argtypes = (
        [_P] * 6 + [_I] * 7 + [_D, _I, _I, _D, _D, _I])
    L.orc_paged_attention_prefill.restype = _I
    L.orc_paged_attention_prefill.argtypes = [_P] * 7 + [_I] * 8 + [_D, _I, _I, _D, _D]
    L.orc_paged_attention_prefill_tree.restype = _I
    L.orc_paged_attention_prefill_tree.argtypes = [_P] * 8 + [_I] * 8 + [_D, _I, _I, _D, _D]


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} returned {rc}")


# ---- codecs -----------------------------------------------------------------
def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Element values (float64) of an array of f16/bf16 (uint16) or E4M3 (uint8) bits."""
    want = np.uint8 if dtype == E4M3 else np.uint16
    bits = np.ascontiguousarray(bits, dtype=want)
    out = np.empty(bits.shape, dtype=np.float64)
    lib().orc_decode_array(_ptr(out), _ptr(bits), bits.size, dtype)
    return out


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().orc_encode_e4m3_array(_ptr(out), _ptr(x), x.size)
    return out


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_elem: int) -> int:
    return int(lib().orc_kv_bytes_per_token(layers, kv_heads, head_dim, bytes_per_elem))


def blocks_for_tokens(n: int, block_size: int = 16) -> int:
    return int(lib().orc_blocks_for_tokens(n, block_size))


# ---- pool -------------------------------------------------------------------
class Pool:
    """Host block pool: free list plus a reference count per block."""

    def __init__(self, num_blocks: int, free_order: np.ndarray | None = None):
        self._order = None if free_order is None else np.ascontiguousarray(free_order, np.int32)
        self.h = lib().orc_pool_create(num_blocks, _ptr(self._order))
        self.num_blocks = num_blocks

    def alloc(self) -> int:
        return lib().orc_pool_alloc(self.h)

    def incref(self, i: int) -> int:
        return lib().orc_pool_incref(self.h, i)

    def decref(self, i: int) -> int:
        return lib().orc_pool_decref(self.h, i)

    def ref_cnt(self, i: int) -> int:
        return lib().orc_pool_ref_cnt(self.h, i)

    def num_free(self) -> int:
        return lib().orc_pool_num_free(self.h)

    def close(self):
        if self.h:
            lib().orc_pool_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Seq:
    """A sequence's block table in a Pool.

    ``caches`` (optional) is a pair of uint8 views of the K and V caches plus
    the byte size of one block; appends then copy shared blocks on write.
    """

    def __init__(self, pool: Pool, block_size: int = 16, _handle=None):
        self.pool = pool
        self.block_size = block_size
        self.h = _handle if _handle is not None else lib().orc_seq_create(pool.h, block_size)

    def append(self, n: int, caches=None) -> np.ndarray:
        slots = np.empty(max(n, 1), dtype=np.int64)
        if caches is None:
            k = v = None
            bb = 0
        else:
            k, v, bb = caches
        rc = lib().orc_seq_append(self.h, n, _ptr(k), _ptr(v), bb, _ptr(slots))
        if rc != 0:
            raise OracleError("block pool exhausted")
        return slots[:n]

    def fork(self) -> "Seq":
        return Seq(self.pool, self.block_size, _handle=lib().orc_seq_fork(self.h))

    @property
    def num_tokens(self) -> int:
        return lib().orc_seq_num_tokens(self.h)

    def table(self) -> np.ndarray:
        n = lib().orc_seq_num_blocks(self.h)
        out = np.empty(max(n, 1), dtype=np.int32)
        lib().orc_seq_table(self.h, _ptr(out), n)
        return out[:n]

    def slot(self, pos: int) -> int:
        return int(lib().orc_seq_slot(self.h, pos))

    def free(self):
        if self.h:
            lib().orc_seq_destroy(self.h)
            self.h = None


# ---- prefix-caching pool ----------------------------------------------------
class CachePool:
    """Block pool with prefix caching: registered full blocks stay matchable at
    reference count 0 until the LRU free queue hands them out again."""

    def __init__(self, num_blocks: int, block_size: int = 16):
        self.h = lib().orc_cpool_create(num_blocks, block_size)
        if not self.h:
            raise OracleError("bad pool arguments")
        self.num_blocks, self.block_size = num_blocks, block_size

    def num_free(self) -> int:
        return lib().orc_cpool_num_free(self.h)

    def num_cached(self) -> int:
        return lib().orc_cpool_num_cached(self.h)

    def ref_cnt(self, i: int) -> int:
        return lib().orc_cpool_ref_cnt(self.h, i)

    def is_cached(self, i: int) -> bool:
        return lib().orc_cpool_is_cached(self.h, i) == 1

    def queue(self) -> np.ndarray:
        out = np.empty(max(self.num_blocks, 1), dtype=np.int32)
        n = lib().orc_cpool_queue(self.h, _ptr(out), self.num_blocks)
        return out[:n]

    def request(self) -> "CacheReq":
        return CacheReq(self, lib().orc_creq_create(self.h))

    def close(self):
        if self.h:
            lib().orc_cpool_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class CacheReq:
    """One request's tokens and block table in a CachePool."""

    def __init__(self, pool: CachePool, handle):
        self.pool, self.h = pool, handle

    def match(self, tokens) -> int:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        m = lib().orc_creq_match(self.h, _ptr(t), len(t))
        if m < 0:
            raise OracleError("match on a request that already holds tokens")
        return m

    def append(self, ids):
        """Returns (slots, cow) where cow is (source, copy) or None; raises
        OracleError (nothing changed) when the pool is out of blocks."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        slots = np.empty(max(len(ids), 1), dtype=np.int64)
        cow = np.empty(2, dtype=np.int32)
        if lib().orc_creq_append(self.h, _ptr(ids), len(ids), _ptr(slots), _ptr(cow)) != 0:
            raise OracleError("block pool exhausted")
        return slots[:len(ids)], (None if cow[0] < 0 else (int(cow[0]), int(cow[1])))

    def fork(self) -> "CacheReq":
        return CacheReq(self.pool, lib().orc_creq_fork(self.h))

    @property
    def num_tokens(self) -> int:
        return lib().orc_creq_num_tokens(self.h)

    def table(self) -> np.ndarray:
        n = lib().orc_creq_table(self.h, None, 0)
        out = np.empty(max(n, 1), dtype=np.int32)
        lib().orc_creq_table(self.h, _ptr(out), n)
        return out[:n]

    def free(self):
        if self.h:
            lib().orc_creq_free(self.h)
            self.h = None


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, pairs, num_blocks: int):
    """In-place copy of whole blocks (source, destination) in both uint8 caches."""
    pr = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    bb = k_cache.nbytes // num_blocks
    _check(lib().orc_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pr), len(pr), num_blocks, bb),
           "orc_copy_blocks")


# ---- cache write and attention ----------------------------------------------
def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, num_blocks, block_size,
                      src_dtype, cache_dtype, k_scale=1.0, v_scale=1.0):
    """In-place write of k, v ([T, Hkv, D] bits) into the uint8 cache buffers."""
    T, hkv, d = k.shape
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    rc = lib().orc_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(slot_mapping), T, hkv, d, block_size, num_blocks,
                                     src_dtype, cache_dtype, k_scale, v_scale)
    _check(rc, "orc_reshape_and_cache")


def paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, num_kv_heads,
                           head_dim, block_size, num_blocks, scale, q_dtype, kv_dtype,
                           k_scale=1.0, v_scale=1.0, partition_size=0) -> np.ndarray:
    S, H, D = q.shape
    assert D == head_dim
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.empty((S, H, D), dtype=np.float64)
    args = [_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(cl), S, H,
            num_kv_heads, D, block_size, bt.shape[1], num_blocks, scale, q_dtype, kv_dtype,
            k_scale, v_scale]
    if partition_size:
        rc = lib().orc_paged_attention_decode_partitioned(*args, partition_size)
    else:
        rc = lib().orc_paged_attention_decode(*args)
    _check(rc, "orc_paged_attention_decode")
    return out


def paged_attention_prefill_tree(q, k_cache, v_cache, block_tables, context_lens,
                                 query_start_loc, tree_mask, num_kv_heads, head_dim, block_size,
                                 num_blocks, scale, q_dtype, kv_dtype, k_scale=1.0,
                                 v_scale=1.0) -> np.ndarray:
    """Tree-masked chunk attention: tree_mask[row] bit j = the chunk key j is
    visible to that query (see orc_paged_attention_prefill_tree)."""
    TQ, H, D = q.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    tm = np.ascontiguousarray(tree_mask, dtype=np.uint64)
    out = np.empty((TQ, H, D), dtype=np.float64)
    rc = lib().orc_paged_attention_prefill_tree(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(cl), _ptr(qsl),
        _ptr(tm), len(cl), TQ, H, num_kv_heads, D, block_size, bt.shape[1], num_blocks, scale,
        q_dtype, kv_dtype, k_scale, v_scale)
    _check(rc, "orc_paged_attention_prefill_tree")
    return out


def paged_attention_prefill(q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                            num_kv_heads, head_dim, block_size, num_blocks, scale, q_dtype,
                            kv_dtype, k_scale=1.0, v_scale=1.0) -> np.ndarray:
    TQ, H, D = q.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    out = np.empty((TQ, H, D), dtype=np.float64)
    rc = lib().orc_paged_attention_prefill(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(cl), _ptr(qsl),
        len(cl), TQ, H, num_kv_heads, D, block_size, bt.shape[1], num_blocks, scale, q_dtype,
        kv_dtype, k_scale, v_scale)
    _check(rc, "orc_paged_attention_prefill")
    return out
