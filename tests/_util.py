"""Shared test helpers: host caches built by the oracle, and an independent
reference (torch scaled_dot_product_attention in float64 on contiguous K/V)
used to pin the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

TORCH_DT = {workloads.F16: torch.float16, workloads.BF16: torch.bfloat16}


def cache_bytes(w) -> int:
    return w.num_blocks * w.num_kv_heads * w.block_size * w.head_dim * w.kv_elem_bytes


def fp8_scale(bits: np.ndarray, dtype: int) -> float:
    """Per-tensor scale amax / 448 (fp32) of a 16-bit tensor, the workloads' choice."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TORCH_DT[dtype])
    return float(np.float32(t.float().abs().max().item()) / np.float32(448.0))


def host_cache(w, k_src, v_src, k_scale=1.0, v_scale=1.0, sentinel=None):
    """Fill uint8 K/V caches with the oracle's cache write: set-up rows, then the
    step's new rows (so the cache holds every context token)."""
    nbytes = cache_bytes(w)
    if sentinel is None:
        kc = np.zeros(nbytes, np.uint8)
        vc = np.zeros(nbytes, np.uint8)
    else:
        kc = np.full(nbytes, sentinel, np.uint8)
        vc = np.full(nbytes, sentinel, np.uint8)
    for rows, slots in ((w.fill_rows, w.fill_slots), (w.new_rows, w.new_slots)):
        if len(rows) == 0:
            continue
        oracle.reshape_and_cache(np.ascontiguousarray(k_src[rows]), np.ascontiguousarray(v_src[rows]),
                                 kc, vc, slots, w.num_blocks, w.block_size, w.src_dtype,
                                 w.kv_dtype, k_scale, v_scale)
    return kc, vc


def to_f64(bits: np.ndarray, dtype: int) -> torch.Tensor:
    """16-bit float bits -> float64 via torch (independent of the oracle codecs)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TORCH_DT[dtype])
    return t.to(torch.float64)


def fp8_dequant_torch(codes: np.ndarray, scale: float) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn)
    return t.to(torch.float64) * scale


def sdpa_ref(q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, scale: float, causal_offset=None):
    """q [Lq, H, D], K/V [Lk, Hkv, D] float64 -> [Lq, H, D].

    Query head h uses KV head h // (H // Hkv).  causal_offset=c lets query i
    see keys 0..c+i; None lets every query see every key."""
    Lq, H, D = q.shape
    Lk, Hkv, _ = K.shape
    g = H // Hkv
    Kx = K.repeat_interleave(g, dim=1).permute(1, 0, 2).unsqueeze(0)
    Vx = V.repeat_interleave(g, dim=1).permute(1, 0, 2).unsqueeze(0)
    qx = q.permute(1, 0, 2).unsqueeze(0)
    mask = None
    if causal_offset is not None:
        i = torch.arange(Lq).unsqueeze(1)
        j = torch.arange(Lk).unsqueeze(0)
        mask = j <= (causal_offset + i)
    if Lk == 0:
        return torch.zeros(Lq, H, D, dtype=torch.float64)
    o = torch.nn.functional.scaled_dot_product_attention(qx, Kx, Vx, attn_mask=mask, scale=scale)
    return o.squeeze(0).permute(1, 0, 2)


def logical_kv_ref(w, k_src, v_src, s, k_scale=1.0, v_scale=1.0):
    """Contiguous [ctx, Hkv, D] float64 K/V of sequence s straight from the source
    rows (through torch's fp8 cast when the cache is E4M3)."""
    rows = w.seq_rows[s]
    if w.kv_dtype == workloads.E4M3:
        ks = to_f64(k_src[rows], w.src_dtype).to(torch.float32)
        vs = to_f64(v_src[rows], w.src_dtype).to(torch.float32)
        kq = (ks / torch.tensor(k_scale, dtype=torch.float32)).to(torch.float8_e4m3fn)
        vq = (vs / torch.tensor(v_scale, dtype=torch.float32)).to(torch.float8_e4m3fn)
        return kq.to(torch.float64) * k_scale, vq.to(torch.float64) * v_scale
    return to_f64(k_src[rows], w.src_dtype), to_f64(v_src[rows], w.src_dtype)


def q_rows(w, s):
    qsl = workloads.query_start_loc(w.q_lens)
    return slice(int(qsl[s]), int(qsl[s + 1]))


def max_rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b) / (np.abs(b) + 1e-12))) if a.size else 0.0
