"""The allocation-free decode entry point, for callers that may not allocate
device memory (a host framework owning every byte through its own pool, or a
loop that must not pay cudaMalloc/cudaFree synchronisation).  It must give the
same output as the workspace entry point, call after call, although every call
reuses the library's one fixed scratch array.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_98_gb300 as pkv
import workloads
from _gpu import TOL_16BIT, TOL_FP8, bits_to_dev, cache_tensors, check_close, decode_inputs, \
    fill_device_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    from paged_kv_cache_98_gb300 import _build
    _build.build()
    pkv.load()


def _setup(w):
    k, v, q = workloads.values_cpu(w)
    # E4M3 caches: a fixed per-tensor scale (N(0,1) values stay below 448 * scale)
    ks = vs = 0.02 if w.kv_dtype == workloads.E4M3 else 1.0
    kc, vc = cache_tensors(w)
    fill_device_cache(w, bits_to_dev(k, w.src_dtype), bits_to_dev(v, w.src_dtype), kc, vc, ks, vs)
    ids, qq, bt, cl = decode_inputs(w, bits_to_dev(q, w.q_dtype))
    return kc, vc, qq, bt, cl, int(w.context_lens[ids].max()), ks, vs


@pytest.mark.parametrize("kv", [workloads.BF16, workloads.E4M3])
def test_noalloc_matches_workspace_entry_two_calls_in_a_row(kv):
    # contexts long enough for several 512-token partitions, so the scratch is used
    w = workloads.independent("noalloc", 61 + kv, [3000, 1, 700, 2600, 1536, 17], 16, 4, 128,
                              workloads.BF16, kv)
    kc, vc, qq, bt, cl, max_ctx, ks, vs = _setup(w)
    assert pkv.decode_workspace_size(qq.shape[0], qq.shape[1], 128, max_ctx) > 0
    tol = TOL_FP8 if kv == workloads.E4M3 else TOL_16BIT
    q2 = torch.flip(qq, dims=[0]).contiguous()  # a second, different query batch
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for query in (qq, q2):
        ref = torch.empty_like(query)
        pkv.paged_attention_decode(ref, query, kc, vc, bt, cl, w.scale, max_context_len=max_ctx,
                                   k_scale=ks, v_scale=vs, device_errors=err)
        got = torch.full_like(query, float("nan"))
        pkv.paged_attention_decode_noalloc(got, query, kc, vc, bt, cl, w.scale, max_ctx,
                                           k_scale=ks, v_scale=vs, device_errors=err)
        torch.cuda.synchronize()
        check_close(got.float().cpu().numpy(), ref.float().cpu().numpy(), tol, "noalloc")
    assert pkv.check_errors(err) == 0


def test_noalloc_rejects_requests_beyond_its_scratch():
    lib = pkv.load()
    limit = 64 * 1024 * 1024
    # 4096 sequences x 32 heads x 8 partitions need far more than the fixed array
    need = pkv.decode_workspace_size(4096, 32, 128, 4096)
    assert need > limit
    rc = lib.pkv_paged_attention_decode_noalloc(
        ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_void_p(512), ctypes.c_void_p(512),
        ctypes.c_void_p(1024), ctypes.c_void_p(2048), 4096, 32, 32, 128, 16, 256, 100000, 4096,
        0.1, 1, 1, 1.0, 1.0, 0, None, None)
    assert rc == -3  # PKV_ERR_WORKSPACE, nothing launched
