"""The oracle's tree-masked chunk attention (speculative verification of a
draft tree), pinned to causal prefill for a chain and to torch
scaled_dot_product_attention (float64, contiguous K/V, an explicit boolean
mask) for random trees."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _util import host_cache, logical_kv_ref, q_rows, to_f64

BF16 = workloads.BF16


def run_tree(w, kc, vc, q, masks):
    return oracle.paged_attention_prefill_tree(q, kc, vc, w.block_tables, w.context_lens,
                                               workloads.query_start_loc(w.q_lens), masks,
                                               w.num_kv_heads, w.head_dim, w.block_size,
                                               w.num_blocks, w.scale, w.q_dtype, w.kv_dtype)


def masked_sdpa(q, K, V, scale, vis):
    """q [Lq, H, D], K/V [Lk, Hkv, D] float64, vis [Lq, Lk] bool -> [Lq, H, D]."""
    H, Hkv = q.shape[1], K.shape[1]
    g = H // Hkv
    Kx = K.repeat_interleave(g, dim=1).permute(1, 0, 2).unsqueeze(0)
    Vx = V.repeat_interleave(g, dim=1).permute(1, 0, 2).unsqueeze(0)
    o = torch.nn.functional.scaled_dot_product_attention(
        q.permute(1, 0, 2).unsqueeze(0), Kx, Vx, attn_mask=vis, scale=scale)
    return o[0].permute(1, 0, 2)


def test_chain_mask_equals_causal_prefill():
    w = workloads.independent("t", 31, [40, 70, 9], 8, 2, 64, BF16, BF16, q_lens=[12, 64, 9])
    k, v, q = workloads.values_cpu(w)
    kc, vc = host_cache(w, k, v)
    masks = np.concatenate([workloads.tree_mask(np.arange(n) - 1) for n in w.q_lens])
    causal = oracle.paged_attention_prefill(q, kc, vc, w.block_tables, w.context_lens,
                                            workloads.query_start_loc(w.q_lens), w.num_kv_heads,
                                            w.head_dim, w.block_size, w.num_blocks, w.scale,
                                            w.q_dtype, w.kv_dtype)
    assert np.array_equal(run_tree(w, kc, vc, q, masks), causal)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_trees_match_masked_sdpa(seed):
    r = np.random.default_rng(seed)
    qlens = [17, 64, 1, 40]
    ctx = [q + int(r.integers(0, 90)) for q in qlens]
    w = workloads.independent("t", 40 + seed, ctx, 8, 2, 64, BF16, BF16, q_lens=qlens)
    k, v, q = workloads.values_cpu(w)
    kc, vc = host_cache(w, k, v)
    masks = []
    for n in qlens:
        parents = workloads.random_tree(r, n)
        if n == 40:
            parents[1:] = 0  # a star: every node a child of the root
        masks.append(workloads.tree_mask(parents))
    masks = np.concatenate(masks)
    out = run_tree(w, kc, vc, q, masks)
    qsl = workloads.query_start_loc(w.q_lens)
    for s in range(w.num_seqs):
        K, V = logical_kv_ref(w, k, v, s)
        rs = q_rows(w, s)
        n, c = int(w.q_lens[s]), int(w.context_lens[s])
        base = c - n
        vis = torch.zeros(n, c, dtype=torch.bool)
        vis[:, :base] = True
        for i in range(n):
            m = int(masks[qsl[s] + i])
            for j in range(n):
                if (m >> j) & 1:
                    vis[i, base + j] = True
        ref = masked_sdpa(to_f64(q[rs], BF16), K, V, w.scale, vis).numpy()
        np.testing.assert_allclose(out[rs], ref, rtol=1e-10, atol=1e-12)


def test_tree_mask_builder():
    parents = np.array([-1, 0, 0, 1, 1, 2])
    m = workloads.tree_mask(parents)
    assert [int(x) for x in m] == [0b1, 0b11, 0b101, 0b1011, 0b10011, 0b100101]


def test_long_chunk_is_rejected():
    w = workloads.independent("t", 50, [80], 4, 2, 64, BF16, BF16, q_lens=[65])
    k, v, q = workloads.values_cpu(w)
    kc, vc = host_cache(w, k, v)
    with pytest.raises(oracle.OracleError):
        run_tree(w, kc, vc, q, np.zeros(65, np.uint64))
