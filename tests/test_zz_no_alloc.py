"""The allocation-free decode entry point, for callers that may not allocate
device memory (a host framework owning every byte through its own pool, or a
loop that must not pay cudaMalloc/cudaFree synchronisation).  It must give the
same output as the workspace entry point and as the CPU oracle, call after
call, although every call reuses the library's one fixed scratch array.

The second call of each pair reads fewer partitions, of other sequences, than
the first wrote, so a read of the previous call's partials or log-sum-exps
from the shared array would show up as a mismatch.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_98_gb300 as pkv
import workloads
from _gpu import TOL_16BIT, TOL_FP8, bits_to_dev, cache_tensors, check_close, fill_device_cache
from _util import host_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    from paged_kv_cache_98_gb300 import _build
    _build.build()
    pkv.load()


@pytest.mark.parametrize("kv", [workloads.BF16, workloads.E4M3])
def test_noalloc_matches_workspace_entry_and_oracle_two_calls_in_a_row(kv):
    # contexts long enough for several 512-token partitions, so the scratch is used
    ctx = [3000, 1, 700, 2600, 1536, 17]
    w = workloads.independent("noalloc", 61 + kv, ctx, 16, 4, 128, workloads.BF16, kv)
    k, v, q = workloads.values_cpu(w)
    # E4M3 caches: a fixed per-tensor scale (N(0,1) values stay below 448 * scale)
    ks = vs = 0.02 if kv == workloads.E4M3 else 1.0
    kc_h, vc_h = host_cache(w, k, v, ks, vs)
    kc, vc = cache_tensors(w)
    fill_device_cache(w, bits_to_dev(k, w.src_dtype), bits_to_dev(v, w.src_dtype), kc, vc, ks, vs)
    qsl = workloads.query_start_loc(w.q_lens)
    ids = w.decode_ids()
    tol = TOL_FP8 if kv == workloads.E4M3 else TOL_16BIT
    # call 1: every sequence, up to 6 partitions each; call 2: three other
    # sequences' queries in another order over shorter contexts (at most 3
    # partitions), rows landing on other slots of the scratch
    calls = [(list(ids), list(w.context_lens[ids])),
             ([ids[4], ids[3], ids[0]], [1100, 900, 600])]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for sel, lens in calls:
        sel = np.asarray(sel)
        lens = np.asarray(lens, np.int32)
        qh = np.ascontiguousarray(q[qsl[sel]])
        query = bits_to_dev(qh, w.q_dtype)
        bt_h = np.ascontiguousarray(w.block_tables[sel])
        bt = torch.from_numpy(bt_h).cuda()
        cl = torch.from_numpy(lens).cuda()
        max_ctx = int(lens.max())
        assert pkv.decode_workspace_size(len(sel), w.num_heads, 128, max_ctx) > 0
        ref = torch.empty_like(query)
        pkv.paged_attention_decode(ref, query, kc, vc, bt, cl, w.scale, max_context_len=max_ctx,
                                   k_scale=ks, v_scale=vs, device_errors=err)
        got = torch.full_like(query, float("nan"))
        pkv.paged_attention_decode_noalloc(got, query, kc, vc, bt, cl, w.scale, max_ctx,
                                           k_scale=ks, v_scale=vs, device_errors=err)
        torch.cuda.synchronize()
        exact = oracle.paged_attention_decode(qh, kc_h, vc_h, bt_h, lens, w.num_kv_heads,
                                              w.head_dim, 16, w.num_blocks, w.scale, w.q_dtype,
                                              w.kv_dtype, ks, vs)
        g = got.float().cpu().numpy()
        check_close(g, ref.float().cpu().numpy(), tol, "noalloc vs workspace entry")
        check_close(g, exact, tol, "noalloc vs oracle")
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
