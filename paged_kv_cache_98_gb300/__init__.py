"""Paged KV-cache attention for one GB300 GPU: Python binding of libpagedkv.so.

Each function here marshals torch tensors into the C ABI declared in
include/pagedkv.h (Python ``X`` is C ``pkv_X``) and launches on the current
torch CUDA stream.  All work runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback: if the library is missing the call raises.

Tensor conventions:
  q, out        [rows, num_heads, head_dim], float16 or bfloat16, contiguous
  k, v          [num_tokens, num_kv_heads, head_dim], float16 or bfloat16
  k_cache,
  v_cache       [num_blocks, num_kv_heads, 16, head_dim]: float16/bfloat16, or
                uint8 / float8_e4m3fn for an E4M3 cache
  block_tables  [num_seqs, max_blocks_per_seq] int32
  context_lens  [num_seqs] int32
  slot_mapping  [num_tokens] int64
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "F16", "BF16", "FP8_E4M3", "PagedKVError", "library_path", "load", "reshape_and_cache",
    "decode_workspace_size", "prefill_workspace_size", "paged_attention_decode",
    "paged_attention_decode_noalloc", "paged_attention_prefill_chunk", "check_errors", "status_string", "version",
    "paged_attention_prefill_tree", "cascade_workspace_size", "paged_attention_decode_cascade",
    "copy_blocks", "BlockPool", "Request", "mixed_workspace_size", "paged_attention_mixed",
    "debug_arm_wait_timeout", "debug_prefill_pairs",
]

F16, BF16, FP8_E4M3 = 0, 1, 2
_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpagedkv.so")
_lib = None
_lock = threading.Lock()

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t


class PagedKVError(RuntimeError):
    """A pkv_* call returned a negative status."""

    def __init__(self, what: str, status: int):
        super().__init__(f"{what} failed: {status_string(status)} ({status})")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load():
    """Loads libpagedkv.so (built by __graft_entry__.build() or _build.build())."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ "
                    "as g; g.build()'); there is no fallback path")
            lib = ctypes.CDLL(_LIB_PATH)
            lib.pkv_version.restype = _I
            lib.pkv_version.argtypes = []
            lib.pkv_status_string.restype = ctypes.c_char_p
            lib.pkv_status_string.argtypes = [_I]
            lib.pkv_reshape_and_cache.restype = _I
            lib.pkv_reshape_and_cache.argtypes = [_P] * 5 + [_I] * 7 + [_F, _F, _P, _P]
            lib.pkv_decode_workspace_size.restype = _SZ
            lib.pkv_decode_workspace_size.argtypes = [_I] * 5
            lib.pkv_prefill_workspace_size.restype = _SZ
            lib.pkv_prefill_workspace_size.argtypes = [_I] * 5
            lib.pkv_paged_attention_decode.restype = _I
            lib.pkv_paged_attention_decode.argtypes = (
                [_P] * 6 + [_I] * 8 + [_F, _I, _I, _F, _F, _I, _P, _SZ, _P, _P])
            lib.pkv_paged_attention_prefill_chunk.restype = _I
            lib.pkv_paged_attention_prefill_chunk.argtypes = (
                [_P] * 7 + [_I] * 10 + [_F, _I, _I, _F, _F, _P, _SZ, _P, _P])
            lib.pkv_paged_attention_decode_noalloc.restype = _I
            lib.pkv_paged_attention_decode_noalloc.argtypes = (
                [_P] * 6 + [_I] * 8 + [_F, _I, _I, _F, _F, _I, _P, _P])
            lib.pkv_paged_attention_prefill_tree.restype = _I
            lib.pkv_paged_attention_prefill_tree.argtypes = (
                [_P] * 8 + [_I] * 10 + [_F, _I, _I, _F, _F, _P, _P])
            lib.pkv_cascade_workspace_size.restype = _SZ
            lib.pkv_cascade_workspace_size.argtypes = [_I] * 5
            lib.pkv_paged_attention_decode_cascade.restype = _I
            lib.pkv_paged_attention_decode_cascade.argtypes = (
                [_P] * 8 + [_I] * 10 + [_F, _I, _I, _F, _F, _P, _SZ, _P, _P])
            lib.pkv_check_errors.restype = _I
            lib.pkv_check_errors.argtypes = [_P, _P, _P]
            lib.pkv_debug_arm_wait_timeout.restype = _I
            lib.pkv_debug_prefill_pairs.restype = _I
            lib.pkv_debug_prefill_pairs.argtypes = [_I]
            lib.pkv_debug_arm_wait_timeout.argtypes = [_I, ctypes.c_uint]
            lib.pkv_mixed_workspace_size.restype = _SZ
            lib.pkv_mixed_workspace_size.argtypes = [_I] * 5
            lib.pkv_paged_attention_mixed.restype = _I
            lib.pkv_paged_attention_mixed.argtypes = (
                [_P] * 7 + [_I] * 11 + [_F, _I, _I, _F, _F, _I, _P, _SZ, _P, _P])
            lib.pkv_copy_blocks.restype = _I
            lib.pkv_copy_blocks.argtypes = [_P, _P, _P] + [_I] * 6 + [_P, _P]
            _I32 = ctypes.c_int32
            lib.pkv_block_pool_create.restype = _I
            lib.pkv_block_pool_create.argtypes = [_I32, _I32, _P]
            lib.pkv_block_pool_destroy.restype = None
            lib.pkv_block_pool_destroy.argtypes = [_P]
            for name in ("pkv_block_pool_num_free", "pkv_block_pool_num_cached",
                         "pkv_request_num_tokens"):
                getattr(lib, name).restype = _I32
                getattr(lib, name).argtypes = [_P]
            for name in ("pkv_block_pool_ref_cnt", "pkv_block_pool_is_cached"):
                getattr(lib, name).restype = _I32
                getattr(lib, name).argtypes = [_P, _I32]
            lib.pkv_block_pool_queue.restype = _I32
            lib.pkv_block_pool_queue.argtypes = [_P, _P, _I32]
            lib.pkv_request_create.restype = _I
            lib.pkv_request_create.argtypes = [_P, _P]
            lib.pkv_request_match_prefix.restype = _I
            lib.pkv_request_match_prefix.argtypes = [_P, _P, _I32, _P]
            lib.pkv_request_append.restype = _I
            lib.pkv_request_append.argtypes = [_P, _P, _I32, _P, _P]
            lib.pkv_request_fork.restype = _I
            lib.pkv_request_fork.argtypes = [_P, _P]
            lib.pkv_request_free.restype = None
            lib.pkv_request_free.argtypes = [_P]
            lib.pkv_request_block_table.restype = _I32
            lib.pkv_request_block_table.argtypes = [_P, _P, _I32]
            lib.pkv_requests_block_tables.restype = _I
            lib.pkv_requests_block_tables.argtypes = [_P, _I32, _I32, _P, _P]
            _lib = lib
    return _lib


def version() -> int:
    return load().pkv_version()


def status_string(status: int) -> str:
    try:
        return load().pkv_status_string(status).decode()
    except Exception:
        return "unknown"


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return FP8_E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must be on the CUDA device")
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _check(what, rc):
    if rc != 0:
        raise PagedKVError(what, rc)


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, k_scale: float = 1.0,
                      v_scale: float = 1.0, device_errors=None, stream=None):
    """Writes k, v ([T, Hkv, D]) into the caches at slot_mapping ([T] int64)."""
    _need_cuda(k, v, k_cache, v_cache, slot_mapping, device_errors)
    T, hkv, d = k.shape
    rc = load().pkv_reshape_and_cache(
        _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), T, hkv, d,
        k_cache.shape[2], k_cache.shape[0], _dtype_code(k), _dtype_code(k_cache), k_scale,
        v_scale, _ptr(device_errors), _stream(stream))
    _check("pkv_reshape_and_cache", rc)


def decode_workspace_size(num_seqs: int, num_heads: int, head_dim: int, max_context_len: int,
                          partition_size: int = 0) -> int:
    return int(load().pkv_decode_workspace_size(num_seqs, num_heads, head_dim, max_context_len,
                                                partition_size))


def prefill_workspace_size(total_q: int, num_heads: int, head_dim: int, max_context_len: int,
                           max_q_len: int) -> int:
    return int(load().pkv_prefill_workspace_size(total_q, num_heads, head_dim, max_context_len,
                                                 max_q_len))


def _workspace(nbytes, workspace, device):
    if nbytes == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                           num_kv_heads: int | None = None, max_context_len: int | None = None,
                           k_scale: float = 1.0, v_scale: float = 1.0, partition_size: int = 0,
                           workspace=None, device_errors=None, stream=None):
    """Decode attention of q ([S, H, D]) over the paged caches into out.

    max_context_len bounds context_lens; passing it avoids a device-to-host read.
    workspace (uint8, >= decode_workspace_size bytes) is allocated if omitted.
    """
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, device_errors)
    S, H, D = q.shape
    nb, hkv, bs, _ = k_cache.shape
    if num_kv_heads is not None and num_kv_heads != hkv:
        raise ValueError("num_kv_heads does not match the cache shape")
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if S else 0
    need = decode_workspace_size(S, H, D, max_context_len, partition_size)
    ws, wsb = _workspace(need, workspace, q.device)
    rc = load().pkv_paged_attention_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        S, H, hkv, D, bs, block_tables.shape[1], nb, max_context_len, scale, _dtype_code(q),
        _dtype_code(k_cache), k_scale, v_scale, partition_size, _ptr(ws), wsb,
        _ptr(device_errors), _stream(stream))
    _check("pkv_paged_attention_decode", rc)
    return out


def paged_attention_prefill_tree(out, q, k_cache, v_cache, block_tables, context_lens,
                                 query_start_loc, tree_mask, scale: float,
                                 max_q_len: int | None = None, max_context_len: int | None = None,
                                 device_errors=None, stream=None):
    """Chunk attention under draft-tree masks (see
    pkv_paged_attention_prefill_tree in include/pagedkv.h): tree_mask is a
    [total_q] int64/uint64 tensor, bit j = the chunk's token j is visible."""
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc, tree_mask,
               device_errors)
    TQ, H, D = q.shape
    nb, hkv, bs, _ = k_cache.shape
    S = query_start_loc.numel() - 1
    if max_q_len is None:
        max_q_len = int((query_start_loc[1:] - query_start_loc[:-1]).max().item()) if S else 0
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if S else 0
    rc = load().pkv_paged_attention_prefill_tree(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(query_start_loc), _ptr(tree_mask), S, TQ, max_q_len, H, hkv, D, bs,
        block_tables.shape[1], nb, max_context_len, scale, _dtype_code(q), _dtype_code(k_cache),
        1.0, 1.0, _ptr(device_errors), _stream(stream))
    _check("pkv_paged_attention_prefill_tree", rc)
    return out


def cascade_workspace_size(num_seqs: int, num_heads: int, head_dim: int, max_context_len: int,
                           max_prefix_len: int) -> int:
    return load().pkv_cascade_workspace_size(num_seqs, num_heads, head_dim, max_context_len,
                                             max_prefix_len)


def paged_attention_decode_cascade(out, q, k_cache, v_cache, block_tables, context_lens,
                                   group_start, prefix_lens, scale: float,
                                   max_context_len: int | None = None,
                                   max_prefix_len: int | None = None, workspace=None,
                                   device_errors=None, stream=None):
    """Decode attention of q ([S, H, D]) over the paged caches into out, reading
    each group's shared prefix once (see pkv_paged_attention_decode_cascade in
    include/pagedkv.h).  group_start: [G + 1] int32; prefix_lens: [S] int32."""
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, group_start, prefix_lens,
               device_errors)
    S, H, D = q.shape
    nb, hkv, bs, _ = k_cache.shape
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if S else 0
    if max_prefix_len is None:
        max_prefix_len = int(prefix_lens.max().item()) if S else 0
    need = cascade_workspace_size(S, H, D, max_context_len, max_prefix_len)
    ws, wsb = _workspace(need, workspace, q.device)
    rc = load().pkv_paged_attention_decode_cascade(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(group_start), _ptr(prefix_lens), S, group_start.numel() - 1, H, hkv, D, bs,
        block_tables.shape[1], nb, max_context_len, max_prefix_len, scale, _dtype_code(q),
        _dtype_code(k_cache), 1.0, 1.0, _ptr(ws), wsb, _ptr(device_errors), _stream(stream))
    _check("pkv_paged_attention_decode_cascade", rc)
    return out


def paged_attention_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens,
                                   scale: float, max_context_len: int, k_scale: float = 1.0,
                                   v_scale: float = 1.0, partition_size: int = 0,
                                   device_errors=None, stream=None):
    """Decode attention with the library's fixed scratch array instead of a
    workspace, for callers that may not allocate device memory (see
    pkv_paged_attention_decode_noalloc in include/pagedkv.h)."""
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, device_errors)
    S, H, D = q.shape
    nb, hkv, bs, _ = k_cache.shape
    # the library takes the scratch array of the current device: make it q's
    with torch.cuda.device(q.device):
        rc = load().pkv_paged_attention_decode_noalloc(
            _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
            _ptr(context_lens), S, H, hkv, D, bs, block_tables.shape[1], nb, max_context_len,
            scale, _dtype_code(q), _dtype_code(k_cache), k_scale, v_scale, partition_size,
            _ptr(device_errors), _stream(stream))
    _check("pkv_paged_attention_decode_noalloc", rc)
    return out


def paged_attention_prefill_chunk(out, q, k_cache, v_cache, block_tables, context_lens,
                                  query_start_loc, scale: float, max_q_len: int | None = None,
                                  max_context_len: int | None = None, k_scale: float = 1.0,
                                  v_scale: float = 1.0, workspace=None, device_errors=None,
                                  stream=None):
    """Causal chunked-prefill attention of q ([total_q, H, D]) into out."""
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
               device_errors)
    TQ, H, D = q.shape
    nb, hkv, bs, _ = k_cache.shape
    S = context_lens.shape[0]
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if S else 0
    if max_q_len is None:
        max_q_len = int((query_start_loc[1:] - query_start_loc[:-1]).max().item()) if S else 0
    need = prefill_workspace_size(TQ, H, D, max_context_len, max_q_len)
    ws, wsb = _workspace(need, workspace, q.device)
    rc = load().pkv_paged_attention_prefill_chunk(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(query_start_loc), S, TQ, max_q_len, H, hkv, D, bs, block_tables.shape[1], nb,
        max_context_len, scale, _dtype_code(q), _dtype_code(k_cache), k_scale, v_scale, _ptr(ws),
        wsb, _ptr(device_errors), _stream(stream))
    _check("pkv_paged_attention_prefill_chunk", rc)
    return out


def mixed_workspace_size(num_decode: int, total_q: int, num_heads: int, head_dim: int,
                         max_context_len: int) -> int:
    return int(load().pkv_mixed_workspace_size(num_decode, total_q, num_heads, head_dim,
                                                max_context_len))


def paged_attention_mixed(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                          num_decode: int, scale: float, max_q_len: int | None = None,
                          max_context_len: int | None = None, k_scale: float = 1.0,
                          v_scale: float = 1.0, prefill_ctas: int = 0, workspace=None,
                          device_errors=None, stream=None):
    """One step's decode rows (the first num_decode sequences, one query row
    each) and prefill chunks (the rest) in one call; see pkv_paged_attention_mixed."""
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
               device_errors)
    TQ, H, D = q.shape
    nb, hkv, bs, _ = k_cache.shape
    S = context_lens.shape[0]
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if S else 0
    if max_q_len is None:
        max_q_len = int((query_start_loc[1:] - query_start_loc[:-1]).max().item()) if S else 0
    need = mixed_workspace_size(num_decode, TQ, H, D, max_context_len)
    ws, wsb = _workspace(need, workspace, q.device)
    rc = load().pkv_paged_attention_mixed(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(query_start_loc), num_decode, S, TQ, max_q_len, H, hkv, D, bs,
        block_tables.shape[1], nb, max_context_len, scale, _dtype_code(q), _dtype_code(k_cache),
        k_scale, v_scale, prefill_ctas, _ptr(ws), wsb, _ptr(device_errors), _stream(stream))
    _check("pkv_paged_attention_mixed", rc)
    return out


def copy_blocks(k_cache, v_cache, block_pairs, device_errors=None, stream=None):
    """Copies whole blocks (block_pairs: [n, 2] int32 on the device, rows
    (source, destination)) in both caches: the copy of copy-on-write."""
    _need_cuda(k_cache, v_cache, block_pairs, device_errors)
    nb, hkv, bs, d = k_cache.shape
    n = block_pairs.shape[0] if block_pairs.dim() == 2 else block_pairs.numel() // 2
    rc = load().pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_pairs), n, hkv, d, bs,
                                nb, _dtype_code(k_cache), _ptr(device_errors), _stream(stream))
    _check("pkv_copy_blocks", rc)


class _Scratch:
    """Host buffers at fixed addresses for the per-token pool calls (token ids
    in, slots and the copy-on-write pair out), grown on demand: each call then
    costs one copy in and one copy out instead of fresh ctypes pointers."""

    def __init__(self):
        import numpy as np
        self.cap = 0
        self.cow = np.empty(2, dtype=np.int32)
        self.cow_addr = self.cow.ctypes.data
        self.matched = ctypes.c_int32()
        self.matched_ref = ctypes.byref(self.matched)
        self.grow(256)

    def grow(self, n: int):
        import numpy as np
        if n <= self.cap:
            return
        self.cap = max(n, 2 * self.cap)
        self.tok = np.empty(self.cap, dtype=np.int32)
        self.slots = np.empty(self.cap, dtype=np.int64)
        self.tok_addr, self.slots_addr = self.tok.ctypes.data, self.slots.ctypes.data


class BlockPool:
    """Host block pool with prefix caching (pkv_block_pool_*): hands out the
    block tables and slot mappings the attention calls consume. Not thread-safe
    (one pool per scheduler thread)."""

    def __init__(self, num_blocks: int, block_size: int = 16):
        h = ctypes.c_void_p()
        lib = load()
        _check("pkv_block_pool_create",
               lib.pkv_block_pool_create(num_blocks, block_size, ctypes.byref(h)))
        self.h, self.num_blocks, self.block_size = h, num_blocks, block_size
        self._live = set()
        self._scratch = _Scratch()
        self._f_append, self._f_match = lib.pkv_request_append, lib.pkv_request_match_prefix

    def num_free(self) -> int:
        return load().pkv_block_pool_num_free(self.h)

    def num_cached(self) -> int:
        return load().pkv_block_pool_num_cached(self.h)

    def ref_cnt(self, block: int) -> int:
        return load().pkv_block_pool_ref_cnt(self.h, block)

    def is_cached(self, block: int) -> bool:
        return load().pkv_block_pool_is_cached(self.h, block) == 1

    def queue(self):
        import numpy as np
        out = np.empty(max(self.num_blocks, 1), dtype=np.int32)
        n = load().pkv_block_pool_queue(self.h, out.ctypes.data_as(ctypes.c_void_p),
                                        self.num_blocks)
        return out[:n]

    def request(self) -> "Request":
        h = ctypes.c_void_p()
        _check("pkv_request_create", load().pkv_request_create(self.h, ctypes.byref(h)))
        return Request(self, h)

    def block_tables(self, requests, max_blocks: int):
        """([n, max_blocks] int32, [n] int32) numpy arrays for a batch of requests."""
        import numpy as np
        arr = (ctypes.c_void_p * max(len(requests), 1))(*[r.h.value for r in requests])
        bt = np.empty((len(requests), max_blocks), dtype=np.int32)
        cl = np.empty(len(requests), dtype=np.int32)
        _check("pkv_requests_block_tables", load().pkv_requests_block_tables(
            ctypes.cast(arr, ctypes.c_void_p), len(requests), max_blocks,
            bt.ctypes.data_as(ctypes.c_void_p), cl.ctypes.data_as(ctypes.c_void_p)))
        return bt, cl

    def close(self):
        for r in list(self._live):
            r.free()
        if self.h:
            load().pkv_block_pool_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Request:
    """One request's tokens and block table in a BlockPool."""

    def __init__(self, pool: BlockPool, handle):
        self.pool, self.h = pool, handle
        pool._live.add(self)

    def match_prefix(self, tokens) -> int:
        sc = self.pool._scratch
        n = len(tokens)
        sc.grow(n)
        sc.tok[:n] = tokens
        _check("pkv_request_match_prefix",
               self.pool._f_match(self.h, sc.tok_addr, n, sc.matched_ref))
        return sc.matched.value

    def append(self, token_ids):
        """Returns (slots int64 numpy array, (source, copy) or None)."""
        sc = self.pool._scratch
        n = len(token_ids)
        sc.grow(n)
        sc.tok[:n] = token_ids
        _check("pkv_request_append",
               self.pool._f_append(self.h, sc.tok_addr, n, sc.slots_addr, sc.cow_addr))
        cow = sc.cow
        return sc.slots[:n].copy(), (None if cow[0] < 0 else (int(cow[0]), int(cow[1])))

    def fork(self) -> "Request":
        h = ctypes.c_void_p()
        _check("pkv_request_fork", load().pkv_request_fork(self.h, ctypes.byref(h)))
        return Request(self.pool, h)

    @property
    def num_tokens(self) -> int:
        return load().pkv_request_num_tokens(self.h)

    def block_table(self):
        import numpy as np
        n = load().pkv_request_block_table(self.h, None, 0)
        out = np.empty(max(n, 1), dtype=np.int32)
        load().pkv_request_block_table(self.h, out.ctypes.data_as(ctypes.c_void_p), n)
        return out[:n]

    def free(self):
        if self.h:
            load().pkv_request_free(self.h)
            self.h = None
            self.pool._live.discard(self)


def debug_arm_wait_timeout(skip_copy: int, wait_limit_us: int = 0) -> None:
    """Test hook: the next attention call's first CTA skips its skip_copy-th
    tile copy and its device waits give up after wait_limit_us, so the call
    reports a wait timeout through its error word (pkv_debug_arm_wait_timeout)."""
    _check("pkv_debug_arm_wait_timeout", load().pkv_debug_arm_wait_timeout(skip_copy,
                                                                            wait_limit_us))


def debug_prefill_pairs(mode: int) -> int:
    """Kernel for causal and draft-tree chunks: 1 CTA pairs, 0 one CTA per
    query tile, 2 (the default) pairs for draft trees only; returns the
    previous setting (pkv_debug_prefill_pairs)."""
    rc = load().pkv_debug_prefill_pairs(int(mode))
    if rc < 0:
        raise PagedKVError("pkv_debug_prefill_pairs", rc)
    return rc


def check_errors(device_errors, stream=None) -> int:
    """Synchronises, reads and clears the device error word; returns its bits."""
    bits = ctypes.c_uint32(0)
    rc = load().pkv_check_errors(_ptr(device_errors), ctypes.byref(bits), _stream(stream))
    if rc not in (0, -5, -6):
        raise PagedKVError("pkv_check_errors", rc)
    return bits.value
