"""Draft-tree chunk attention (pkv_paged_attention_prefill_tree) vs the CPU
oracle's tree-masked attention: |gpu - ref| <= 2e-3 + 1e-2 |ref|."""
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
    torch.cuda.init()


def all_inputs(w, q_all):
    """Every sequence's queries (chunks of any length, single tokens included)."""
    dev = q_all.device
    bt = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(dev)
    cl = torch.from_numpy(np.ascontiguousarray(w.context_lens)).to(dev)
    qsl = torch.from_numpy(workloads.query_start_loc(w.q_lens)).to(dev)
    return q_all.contiguous(), bt, cl, qsl


def run_tree(w, masks, sentinel=0xFF):
    k, v, q = workloads.values_cpu(w)
    kc_h, vc_h = host_cache(w, k, v)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc, vc = cache_tensors(w, sentinel=sentinel)
    fill_device_cache(w, bits_to_dev(k, w.src_dtype), bits_to_dev(v, w.src_dtype), kc, vc,
                      errors=err)
    qq, bt, cl, qsl_d = all_inputs(w, bits_to_dev(q, w.q_dtype))
    out = torch.empty_like(qq)
    tm = torch.from_numpy(masks.view(np.int64)).cuda()
    pkv.paged_attention_prefill_tree(out, qq, kc, vc, bt, cl, qsl_d, tm, w.scale,
                                     device_errors=err)
    assert pkv.check_errors(err) == 0
    ref = oracle.paged_attention_prefill_tree(np.ascontiguousarray(q), kc_h, vc_h, w.block_tables,
                                              w.context_lens, workloads.query_start_loc(w.q_lens),
                                              masks, w.num_kv_heads, w.head_dim, 16, w.num_blocks,
                                              w.scale, w.q_dtype, w.kv_dtype)
    check_close(out.float().cpu().numpy(), ref, tol(w), f"{w.name} tree")
    return out, ref


@pytest.mark.parametrize("g,dt", [(4, BF16), (8, F16), (1, BF16), (2, BF16)])
def test_random_draft_trees(g, dt):
    r = np.random.default_rng(7 + g)
    qlens = [64, 7, 33, 1, 20]
    prior = [300, 0, 16, 1000, 2049]
    w = workloads.independent("tree", 60 + g, [a + b for a, b in zip(qlens, prior)], 2 * g, 2,
                              128, dt, dt, q_lens=qlens)
    masks = []
    for n in qlens:
        parents = workloads.random_tree(r, n)
        if n == 33:
            parents[1:] = 0  # a star
        masks.append(workloads.tree_mask(parents))
    run_tree(w, np.concatenate(masks))


@pytest.mark.parametrize("pairs", [1, 0])
def test_chain_equals_causal_chunk(pairs):
    """A chain-shaped tree is the causal chunk: on the same kernel (CTA pairs,
    or one CTA per tile) the same arithmetic, so the same bytes, and both meet
    the tolerance against the oracle."""
    prev = pkv.debug_prefill_pairs(pairs)
    try:
        qlens = [64, 30]
        w = workloads.independent("tree-chain", 70, [600, 95], 16, 2, 128, BF16, BF16,
                                  q_lens=qlens)
        masks = np.concatenate([workloads.tree_mask(np.arange(n) - 1) for n in qlens])
        out_t, ref = run_tree(w, masks)
        k, v, q = workloads.values_cpu(w)
        kc, vc = cache_tensors(w)
        fill_device_cache(w, bits_to_dev(k, BF16), bits_to_dev(v, BF16), kc, vc)
        qq, bt, cl, qsl_d = all_inputs(w, bits_to_dev(q, BF16))
        out_c = torch.empty_like(qq)
        pkv.paged_attention_prefill_chunk(out_c, qq, kc, vc, bt, cl, qsl_d, w.scale,
                                          max_q_len=64, max_context_len=600)
        check_close(out_c.float().cpu().numpy(), ref, tol(w), "causal chunk")
        assert torch.equal(out_t.view(torch.int16), out_c.view(torch.int16))
    finally:
        pkv.debug_prefill_pairs(prev)


def test_unsupported_and_invalid():
    w = workloads.independent("tree-x", 71, [80], 8, 2, 128, BF16, BF16, q_lens=[65])
    k, v, q = workloads.values_cpu(w)
    kc, vc = cache_tensors(w)
    qq, bt, cl, qsl_d = all_inputs(w, bits_to_dev(q, BF16))
    out = torch.empty_like(qq)
    tm = torch.zeros(65, dtype=torch.int64, device="cuda")
    with pytest.raises(pkv.PagedKVError):  # a chunk longer than 64
        pkv.paged_attention_prefill_tree(out, qq, kc, vc, bt, cl, qsl_d, tm, w.scale)


def test_full_size_draft_trees_sampled():
    """A verification batch at serving size: 128 sequences with the 70B-GQA head
    shape (64 q / 8 kv heads), contexts drawn like that workload's, each with a
    random 64-token draft tree.  Every output is finite; sampled sequences (the
    shortest and the longest context, and three more) match the oracle, each
    computed from a compact cache of its own rows."""
    r = np.random.default_rng(77)
    prior = np.clip(np.exp(r.normal(np.log(2000.0), 1.0, size=128)).astype(int), 16, 12000)
    qlens = [64] * 128
    w = workloads.independent("tree-full", 78, list(prior + 64), 64, 8, 128, BF16, BF16,
                              q_lens=qlens)
    masks = np.concatenate([workloads.tree_mask(workloads.random_tree(r, 64)) for _ in qlens])
    dev = "cuda"
    k, v, q = workloads.values_device(w, dev)
    kc, vc = cache_tensors(w)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    fill_device_cache(w, k, v, kc, vc, errors=err)
    qq, bt, cl, qsl_d = all_inputs(w, q)
    out = torch.empty_like(qq)
    pkv.paged_attention_prefill_tree(out, qq, kc, vc, bt, cl, qsl_d,
                                     torch.from_numpy(masks.view(np.int64)).cuda(), w.scale,
                                     max_q_len=64, max_context_len=int(w.context_lens.max()),
                                     device_errors=err)
    assert pkv.check_errors(err) == 0
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    qsl = workloads.query_start_loc(w.q_lens)
    bits = lambda t: t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    for s in sorted({int(np.argmin(prior)), int(np.argmax(prior)), 0, 57, 127}):
        rows = torch.from_numpy(w.seq_rows[s]).to(dev)
        c = len(w.seq_rows[s])
        nb = -(-c // 16)
        kc_h = np.zeros(nb * 8 * 16 * 128 * 2, np.uint8)
        vc_h = np.zeros_like(kc_h)
        oracle.reshape_and_cache(bits(k.index_select(0, rows)), bits(v.index_select(0, rows)),
                                 kc_h, vc_h, np.arange(c, dtype=np.int64), nb, 16, BF16, BF16)
        ref = oracle.paged_attention_prefill_tree(
            bits(q[int(qsl[s]):int(qsl[s + 1])]), kc_h, vc_h,
            np.arange(nb, dtype=np.int32)[None], np.array([c], np.int32),
            np.array([0, 64], np.int32), masks[qsl[s]:qsl[s + 1]], 8, 128, 16, nb, w.scale,
            BF16, BF16)
        check_close(got[qsl[s]:qsl[s + 1]], ref, tol(w), f"tree sequence {s}")
