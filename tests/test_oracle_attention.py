"""Oracle attention pinned to an independent library routine (torch
scaled_dot_product_attention, float64, contiguous K/V), to closed-form special
cases, and to the layout invariants of the paged cache."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _util import (fp8_dequant_torch, fp8_scale, host_cache, logical_kv_ref, q_rows, sdpa_ref,
                   to_f64)

F16, BF16, E4M3 = workloads.F16, workloads.BF16, workloads.E4M3
CTXS = [1, 15, 16, 17, 31, 32, 33, 100]


def run_decode(w, kc, vc, q, k_scale=1.0, v_scale=1.0, partition_size=0, tables=None):
    ids = w.decode_ids()
    qq = np.ascontiguousarray(q[[q_rows(w, s).start for s in ids]])
    bt = w.block_tables[ids] if tables is None else tables
    return oracle.paged_attention_decode(qq, kc, vc, bt, w.context_lens[ids], w.num_kv_heads,
                                         w.head_dim, w.block_size, w.num_blocks, w.scale,
                                         w.q_dtype, w.kv_dtype, k_scale, v_scale, partition_size)


def check_against_sdpa(w, out, k, v, q, k_scale=1.0, v_scale=1.0):
    for i, s in enumerate(w.decode_ids()):
        K, V = logical_kv_ref(w, k, v, s, k_scale, v_scale)
        qs = to_f64(q[q_rows(w, s)], w.q_dtype)
        ref = sdpa_ref(qs, K, V, w.scale).numpy()[0]
        np.testing.assert_allclose(out[i], ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_matches_sdpa(g, D):
    hkv = 2
    w = workloads.independent("p", 100 + g + D, CTXS, hkv * g, hkv, D, BF16, BF16)
    k, v, q = workloads.values_cpu(w)
    kc, vc = host_cache(w, k, v)
    out = run_decode(w, kc, vc, q)
    check_against_sdpa(w, out, k, v, q)


def test_tiny_workload_matches_sdpa():
    for seed in range(3):
        w = workloads.tiny(seed)
        k, v, q = workloads.values_cpu(w)
        kc, vc = host_cache(w, k, v)
        check_against_sdpa(w, run_decode(w, kc, vc, q), k, v, q)


def test_cache_write_places_every_token():
    w = workloads.independent("p", 7, CTXS, 4, 2, 64, F16, F16)
    k, v, q = workloads.values_cpu(w)
    kc, vc = host_cache(w, k, v, sentinel=0xA5)
    K = kc.view(np.uint16).reshape(w.num_blocks, w.num_kv_heads, 16, w.head_dim)
    V = vc.view(np.uint16).reshape(w.num_blocks, w.num_kv_heads, 16, w.head_dim)
    touched = np.zeros((w.num_blocks, 16), bool)
    for s in range(w.num_seqs):
        for pos, row in enumerate(w.seq_rows[s]):
            b = w.block_tables[s, pos // 16]
            assert np.array_equal(K[b, :, pos % 16], k[row])
            assert np.array_equal(V[b, :, pos % 16], v[row])
            touched[b, pos % 16] = True
    # every other slot keeps the sentinel
    untouched = ~touched
    assert np.all(K.transpose(0, 2, 1, 3)[untouched] == 0xA5A5)
    assert np.all(V.transpose(0, 2, 1, 3)[untouched] == 0xA5A5)


def test_single_token_context_returns_v0():
    w = workloads.independent("p", 8, [1, 1, 1], 4, 2, 64, BF16, BF16)
    k, v, q = workloads.values_cpu(w)
    kc, vc = host_cache(w, k, v)
    out = run_decode(w, kc, vc, q)
    for s in range(3):
        v0 = oracle.decode(v[w.seq_rows[s][0]], BF16)  # [Hkv, D]
        assert np.array_equal(out[s], np.repeat(v0, 2, axis=0))


def test_identical_keys_give_mean_of_values():
    w = workloads.independent("p", 9, [37, 64], 2, 1, 64, BF16, BF16)
    k, v, q = workloads.values_cpu(w)
    k[:] = k[0]
    kc, vc = host_cache(w, k, v)
    out = run_decode(w, kc, vc, q)
    for s in range(2):
        mean = oracle.decode(v[w.seq_rows[s]], BF16).mean(axis=0)  # [Hkv, D]
        np.testing.assert_allclose(out[s], np.repeat(mean, 2, axis=0), rtol=1e-12, atol=1e-14)


def test_dominant_key_selects_its_value():
    w = workloads.independent("p", 10, [50], 1, 1, 64, F16, F16)
    k, v, q = workloads.values_cpu(w)
    q[:] = np.float16(1.0).view(np.uint16)
    k[:] = np.float16(0.0).view(np.uint16)
    j = 23
    k[w.seq_rows[0][j]] = np.float16(4.0).view(np.uint16)  # score 8*4*64 = 32 above the rest
    kc, vc = host_cache(w, k, v)
    out = run_decode(w, kc, vc, q)
    vj = oracle.decode(v[w.seq_rows[0][j]], F16)[0]
    np.testing.assert_allclose(out[0, 0], vj, rtol=0, atol=1e-12 + 49 * np.exp(-32.0) * 10)


def test_empty_context_gives_zeros():
    w = workloads.independent("p", 11, [5, 20], 2, 2, 64, BF16, BF16)
    k, v, q = workloads.values_cpu(w)
    kc, vc = host_cache(w, k, v)
    ctx = w.context_lens.copy()
    ctx[0] = 0
    out = oracle.paged_attention_decode(np.ascontiguousarray(q[:2]), kc, vc, w.block_tables, ctx,
                                        2, 64, 16, w.num_blocks, w.scale, BF16, BF16)
    assert np.all(out[0] == 0.0)


def test_block_permutation_leaves_output_bit_identical():
    w = workloads.independent("p", 12, CTXS, 8, 2, 64, BF16, BF16)
    k, v, q = workloads.values_cpu(w)
    kc, vc = host_cache(w, k, v)
    out = run_decode(w, kc, vc, q)
    perm = workloads.rng(99).permutation(w.num_blocks)
    bb = w.num_kv_heads * 16 * w.head_dim * 2
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    for b in range(w.num_blocks):
        kc2[perm[b] * bb:(perm[b] + 1) * bb] = kc[b * bb:(b + 1) * bb]
        vc2[perm[b] * bb:(perm[b] + 1) * bb] = vc[b * bb:(b + 1) * bb]
    tables = perm[w.block_tables].astype(np.int32)
    out2 = run_decode(w, kc2, vc2, q, tables=tables)
    assert np.array_equal(out, out2)


def test_shared_prefix_equals_unshared_copies():
    w = workloads.shared_prefix("s", 13, [37, 64, 5], [[3, 20, 1], [5, 40], [2]], 8, 2, 64,
                                BF16, BF16)
    k, v, q = workloads.values_cpu(w)
    kc, vc = host_cache(w, k, v)
    out = run_decode(w, kc, vc, q)
    # deep copies: every sequence gets private blocks holding the same bytes
    bb = w.num_kv_heads * 16 * w.head_dim * 2
    nblocks = [-(-int(c) // 16) for c in w.context_lens]
    total = sum(nblocks)
    kc2 = np.zeros(total * bb, np.uint8)
    vc2 = np.zeros(total * bb, np.uint8)
    tables = np.zeros((w.num_seqs, max(nblocks)), np.int32)
    nxt = 0
    for s in range(w.num_seqs):
        for j in range(nblocks[s]):
            b = w.block_tables[s, j]
            kc2[nxt * bb:(nxt + 1) * bb] = kc[b * bb:(b + 1) * bb]
            vc2[nxt * bb:(nxt + 1) * bb] = vc[b * bb:(b + 1) * bb]
            tables[s, j] = nxt
            nxt += 1
    qq = np.ascontiguousarray(q)
    out2 = oracle.paged_attention_decode(qq, kc2, vc2, tables, w.context_lens, w.num_kv_heads,
                                         w.head_dim, 16, total, w.scale, BF16, BF16)
    assert np.array_equal(out, out2)
    check_against_sdpa(w, out, k, v, q)


@pytest.mark.parametrize("psize", [16, 32, 64, 512])
def test_partitioned_equals_single_pass(psize):
    w = workloads.independent("p", 14, [1, 16, 17, 100, 300, 513], 4, 2, 64, BF16, BF16)
    k, v, q = workloads.values_cpu(w)
    kc, vc = host_cache(w, k, v)
    a = run_decode(w, kc, vc, q)
    b = run_decode(w, kc, vc, q, partition_size=psize)
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-14)


def test_fp8_cache_write_matches_torch_cast():
    w = workloads.independent("p", 15, CTXS, 8, 2, 128, BF16, E4M3)
    k, v, q = workloads.values_cpu(w)
    ks, vs = fp8_scale(k, BF16), fp8_scale(v, BF16)
    kc, vc = host_cache(w, k, v, ks, vs)
    K = kc.reshape(w.num_blocks, w.num_kv_heads, 16, w.head_dim)
    for s in range(w.num_seqs):
        rows = w.seq_rows[s]
        x = to_f64(k[rows], BF16).to(torch.float32)
        ref = (x / torch.tensor(ks, dtype=torch.float32)).to(torch.float8_e4m3fn)
        ref = ref.view(torch.uint8).numpy()
        for pos in range(len(rows)):
            b = w.block_tables[s, pos // 16]
            assert np.array_equal(K[b, :, pos % 16], ref[pos])


def test_fp8_decode_matches_sdpa_on_dequantized():
    w = workloads.independent("p", 16, CTXS, 8, 2, 128, BF16, E4M3)
    k, v, q = workloads.values_cpu(w)
    ks, vs = fp8_scale(k, BF16), fp8_scale(v, BF16)
    kc, vc = host_cache(w, k, v, ks, vs)
    out = run_decode(w, kc, vc, q, ks, vs)
    check_against_sdpa(w, out, k, v, q, ks, vs)
    # dequantisation through torch's own float8 type agrees with the cache bytes
    deq = fp8_dequant_torch(kc[:64], ks).numpy()
    np.testing.assert_array_equal(deq, oracle.decode(kc[:64], E4M3) * ks)


def run_prefill(w, kc, vc, q, k_scale=1.0, v_scale=1.0):
    return oracle.paged_attention_prefill(q, kc, vc, w.block_tables, w.context_lens,
                                          workloads.query_start_loc(w.q_lens), w.num_kv_heads,
                                          w.head_dim, w.block_size, w.num_blocks, w.scale,
                                          w.q_dtype, w.kv_dtype, k_scale, v_scale)


@pytest.mark.parametrize("g", [1, 4])
def test_prefill_matches_causal_sdpa(g):
    ctx = [40, 17, 64, 100]
    qlen = [40, 5, 33, 1]
    w = workloads.independent("p", 17 + g, ctx, 2 * g, 2, 64, BF16, BF16, q_lens=qlen)
    k, v, q = workloads.values_cpu(w)
    kc, vc = host_cache(w, k, v)
    out = run_prefill(w, kc, vc, q)
    for s in range(w.num_seqs):
        K, V = logical_kv_ref(w, k, v, s)
        rs = q_rows(w, s)
        ref = sdpa_ref(to_f64(q[rs], BF16), K, V, w.scale,
                       causal_offset=int(w.context_lens[s] - w.q_lens[s])).numpy()
        np.testing.assert_allclose(out[rs], ref, rtol=1e-10, atol=1e-12)


def test_prefill_with_one_query_equals_decode():
    w = workloads.independent("p", 19, CTXS, 8, 2, 64, BF16, BF16)
    k, v, q = workloads.values_cpu(w)
    kc, vc = host_cache(w, k, v)
    assert np.array_equal(run_prefill(w, kc, vc, q), run_decode(w, kc, vc, q))


def test_bad_arguments_are_rejected():
    w = workloads.tiny(0)
    k, v, q = workloads.values_cpu(w)
    kc, vc = host_cache(w, k, v)
    with pytest.raises(oracle.OracleError):  # H not a multiple of Hkv
        oracle.paged_attention_decode(np.ascontiguousarray(q), kc, vc, w.block_tables,
                                      w.context_lens, 3, 64, 16, w.num_blocks, w.scale, F16, F16)
    bad = w.block_tables.copy()
    bad[0, 0] = w.num_blocks  # outside the pool
    with pytest.raises(oracle.OracleError):
        oracle.paged_attention_decode(np.ascontiguousarray(q), kc, vc, bad, w.context_lens, 4, 64,
                                      16, w.num_blocks, w.scale, F16, F16)
    with pytest.raises(oracle.OracleError):  # duplicate slot
        oracle.reshape_and_cache(k[:2], v[:2], kc, vc, np.array([3, 3]), w.num_blocks, 16, F16, F16)
