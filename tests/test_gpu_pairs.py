"""Causal and draft-tree chunks on CTA pairs (two CTAs share each 256-row
query tile) against the single-CTA kernel and the CPU oracle.

The two kernels compute the same per-row products and softmax in the same
order, so their outputs must agree bit for bit; each must also meet the
tolerance against the oracle on its own (|gpu - ref| <= 2e-3 + 1e-2 |ref|)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_98_gb300 as pkv
import workloads
from _gpu import bits_to_dev, cache_tensors, check_close, fill_device_cache, tol
from _util import host_cache

pytestmark = pytest.mark.gpu
F16, BF16 = workloads.F16, workloads.BF16


@pytest.fixture(scope="module", autouse=True)
def _library():
    from paged_kv_cache_98_gb300 import _build
    _build.build()
    pkv.load()
    prev = pkv.debug_prefill_pairs(0)
    yield
    pkv.debug_prefill_pairs(prev)


def _both(w, call):
    """call() on the device state of w with CTA pairs and with one CTA per tile."""
    outs = []
    for mode in (1, 0):
        pkv.debug_prefill_pairs(mode)
        outs.append(call())
    return outs


def _state(w, sentinel=None):
    k, v, q = workloads.values_cpu(w)
    kc_h, vc_h = host_cache(w, k, v)
    kc, vc = cache_tensors(w, sentinel=sentinel)
    fill_device_cache(w, bits_to_dev(k, w.src_dtype), bits_to_dev(v, w.src_dtype), kc, vc)
    dev = "cuda"
    bt = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(dev)
    cl = torch.from_numpy(np.ascontiguousarray(w.context_lens)).to(dev)
    qsl = torch.from_numpy(workloads.query_start_loc(w.q_lens)).to(dev)
    return q, kc_h, vc_h, kc, vc, bits_to_dev(q, w.q_dtype), bt, cl, qsl


@pytest.mark.parametrize("g,dt", [(1, BF16), (2, F16), (4, BF16), (8, BF16), (16, F16)])
def test_causal_chunks_pairs_equal_single(g, dt):
    # chunks of many lengths (1 .. 700 queries), prior contexts with partial last blocks
    qlens = [700, 1, 33, 257, 64, 129]
    prior = [1100, 5, 0, 2000, 31, 600]
    w = workloads.independent("pairs", 8100 + g, [a + b for a, b in zip(qlens, prior)], 2 * g, 2,
                              128, dt, dt, q_lens=qlens)
    q, kc_h, vc_h, kc, vc, qd, bt, cl, qsl = _state(w, sentinel=0xFF)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call():
        out = torch.empty_like(qd)
        pkv.paged_attention_prefill_chunk(out, qd, kc, vc, bt, cl, qsl, w.scale,
                                          max_q_len=max(qlens),
                                          max_context_len=int(w.context_lens.max()),
                                          device_errors=err)
        return out

    pair, single = _both(w, call)
    assert pkv.check_errors(err) == 0
    ref = oracle.paged_attention_prefill(np.ascontiguousarray(q), kc_h, vc_h, w.block_tables,
                                         w.context_lens, workloads.query_start_loc(w.q_lens),
                                         w.num_kv_heads, w.head_dim, 16, w.num_blocks, w.scale,
                                         w.q_dtype, w.kv_dtype)
    check_close(pair.float().cpu().numpy(), ref, tol(w), "pairs")
    check_close(single.float().cpu().numpy(), ref, tol(w), "single CTAs")
    assert torch.equal(pair.view(torch.int16), single.view(torch.int16))


@pytest.mark.parametrize("g", [4, 8])
def test_draft_trees_pairs_equal_single(g):
    r = np.random.default_rng(300 + g)
    qlens = [64, 64, 17, 40]
    prior = [900, 12, 2050, 300]
    w = workloads.independent("pairs-tree", 8200 + g, [a + b for a, b in zip(qlens, prior)],
                              2 * g, 2, 128, BF16, BF16, q_lens=qlens)
    masks = np.concatenate([workloads.tree_mask(workloads.random_tree(r, n)) for n in qlens])
    q, kc_h, vc_h, kc, vc, qd, bt, cl, qsl = _state(w, sentinel=0xFF)
    tm = torch.from_numpy(masks.view(np.int64)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call():
        out = torch.empty_like(qd)
        pkv.paged_attention_prefill_tree(out, qd, kc, vc, bt, cl, qsl, tm, w.scale,
                                         device_errors=err)
        return out

    pair, single = _both(w, call)
    assert pkv.check_errors(err) == 0
    ref = oracle.paged_attention_prefill_tree(np.ascontiguousarray(q), kc_h, vc_h, w.block_tables,
                                              w.context_lens, workloads.query_start_loc(w.q_lens),
                                              masks, w.num_kv_heads, w.head_dim, 16, w.num_blocks,
                                              w.scale, w.q_dtype, w.kv_dtype)
    check_close(pair.float().cpu().numpy(), ref, tol(w), "pairs tree")
    check_close(single.float().cpu().numpy(), ref, tol(w), "single-CTA tree")
    assert torch.equal(pair.view(torch.int16), single.view(torch.int16))


def test_pairs_wait_runs_out():
    """The device-wait timeout on the pair kernel: the even CTA of the first
    pair skips one copy, both CTAs give up, and the next call is correct."""
    qlens = [300, 128]
    w = workloads.independent("pairs-timeout", 8300, [1300, 700], 16, 4, 128, BF16, BF16,
                              q_lens=qlens)
    q, kc_h, vc_h, kc, vc, qd, bt, cl, qsl = _state(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(qd)
    pkv.debug_prefill_pairs(1)
    pkv.debug_arm_wait_timeout(3, 20000)
    pkv.paged_attention_prefill_chunk(out, qd, kc, vc, bt, cl, qsl, w.scale, max_q_len=300,
                                      max_context_len=1300, device_errors=err)
    assert pkv.check_errors(err) & 0x8
    pkv.paged_attention_prefill_chunk(out, qd, kc, vc, bt, cl, qsl, w.scale, max_q_len=300,
                                      max_context_len=1300, device_errors=err)
    assert pkv.check_errors(err) == 0
    ref = oracle.paged_attention_prefill(np.ascontiguousarray(q), kc_h, vc_h, w.block_tables,
                                         w.context_lens, workloads.query_start_loc(w.q_lens),
                                         w.num_kv_heads, w.head_dim, 16, w.num_blocks, w.scale,
                                         w.q_dtype, w.kv_dtype)
    check_close(out.float().cpu().numpy(), ref, tol(w), "pairs after a timeout")
