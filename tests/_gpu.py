"""GPU-side helpers for the parity tests: device caches filled through the
library's own cache write, and the benchmark spec's tolerances."""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_98_gb300 as pkv
import workloads

TD = {workloads.F16: torch.float16, workloads.BF16: torch.bfloat16}

# |gpu - ref| <= ATOL + RTOL * |ref|, elementwise
TOL_16BIT = (2e-3, 1e-2)
TOL_FP8 = (3e-2, 5e-2)


def tol(w):
    return TOL_FP8 if w.kv_dtype == workloads.E4M3 else TOL_16BIT


def bits_to_dev(bits: np.ndarray, dtype: int, dev="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(TD[dtype]).to(dev)


def cache_tensors(w, dev="cuda", sentinel: int | None = None):
    shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    if w.kv_dtype == workloads.E4M3:
        kc = torch.empty(shape, dtype=torch.uint8, device=dev)
        vc = torch.empty(shape, dtype=torch.uint8, device=dev)
    else:
        kc = torch.empty(shape, dtype=TD[w.kv_dtype], device=dev)
        vc = torch.empty(shape, dtype=TD[w.kv_dtype], device=dev)
    if sentinel is not None:
        kc.view(torch.uint8).fill_(sentinel)
        vc.view(torch.uint8).fill_(sentinel)
    else:
        kc.view(torch.uint8).zero_()
        vc.view(torch.uint8).zero_()
    return kc, vc


def fill_device_cache(w, k_src, v_src, kc, vc, k_scale=1.0, v_scale=1.0, errors=None,
                      include_new=True):
    """Writes every context token into the device caches with the library's cache write."""
    dev = kc.device
    parts = [(w.fill_rows, w.fill_slots)]
    if include_new:
        parts.append((w.new_rows, w.new_slots))
    for rows, slots in parts:
        if len(rows) == 0:
            continue
        r = torch.from_numpy(rows).to(dev)
        ks = k_src.index_select(0, r).contiguous()
        vs = v_src.index_select(0, r).contiguous()
        pkv.reshape_and_cache(ks, vs, kc, vc, torch.from_numpy(slots).to(dev), k_scale, v_scale,
                              device_errors=errors)


def check_close(gpu: np.ndarray, ref: np.ndarray, atol_rtol, what=""):
    atol, rtol = atol_rtol
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    err = np.abs(gpu - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; first at {tuple(i)}: "
            f"gpu {gpu[tuple(i)]!r} ref {ref[tuple(i)]!r} (max err {err.max():.3g})")


def decode_inputs(w, q_all: torch.Tensor):
    """q rows, block tables and context lengths of the workload's decode sequences."""
    ids = w.decode_ids()
    qsl = workloads.query_start_loc(w.q_lens)
    dev = q_all.device
    q = q_all.index_select(0, torch.from_numpy(qsl[ids].astype(np.int64)).to(dev)).contiguous()
    bt = torch.from_numpy(np.ascontiguousarray(w.block_tables[ids])).to(dev)
    cl = torch.from_numpy(np.ascontiguousarray(w.context_lens[ids])).to(dev)
    return ids, q, bt, cl


def prefill_inputs(w, q_all: torch.Tensor):
    ids = w.prefill_ids()
    qsl = workloads.query_start_loc(w.q_lens)
    dev = q_all.device
    rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in ids]).astype(np.int64)
    q = q_all.index_select(0, torch.from_numpy(rows).to(dev)).contiguous()
    bt = torch.from_numpy(np.ascontiguousarray(w.block_tables[ids])).to(dev)
    cl = torch.from_numpy(np.ascontiguousarray(w.context_lens[ids])).to(dev)
    sub_qsl = workloads.query_start_loc(w.q_lens[ids])
    return ids, q, bt, cl, torch.from_numpy(sub_qsl).to(dev)
