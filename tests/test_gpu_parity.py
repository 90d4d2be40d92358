"""CUDA path vs the CPU oracle, through the C ABI (Python binding).

Cache writes must be bit-exact over the whole cache buffer; attention must be
within |gpu - ref| <= 2e-3 + 1e-2 |ref| (fp16/bf16 caches) or
3e-2 + 5e-2 |ref| (E4M3 caches), elementwise.  The oracle never sees a byte
the CUDA path produced: it builds its own cache from the same seeded source
rows with its own cache write.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_98_gb300 as pkv
import workloads
from _gpu import (bits_to_dev, cache_tensors, check_close, decode_inputs, fill_device_cache,
                  prefill_inputs, tol)
from _util import cache_bytes, fp8_scale, host_cache

pytestmark = pytest.mark.gpu
F16, BF16, E4M3 = workloads.F16, workloads.BF16, workloads.E4M3


@pytest.fixture(scope="module", autouse=True)
def _library():
    from paged_kv_cache_98_gb300 import _build
    _build.build()
    pkv.load()
    torch.cuda.init()


def errors_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def run_case(w, partition_size=0, sentinel=None):
    """Fills both caches, runs the workload's decode and prefill rows on both
    sides and compares them; returns the number of compared elements."""
    k, v, q = workloads.values_cpu(w)
    ks = vs = 1.0
    if w.kv_dtype == E4M3:
        ks, vs = fp8_scale(k, w.src_dtype), fp8_scale(v, w.src_dtype)
    kc_h, vc_h = host_cache(w, k, v, ks, vs, sentinel=sentinel)
    err = errors_word()
    kd, vd = bits_to_dev(k, w.src_dtype), bits_to_dev(v, w.src_dtype)
    qd = bits_to_dev(q, w.q_dtype)
    kc, vc = cache_tensors(w, sentinel=sentinel)
    fill_device_cache(w, kd, vd, kc, vc, ks, vs, errors=err)
    # the cache write is bit-exact over the whole buffer
    assert np.array_equal(kc.view(torch.uint8).cpu().numpy().reshape(-1), kc_h)
    assert np.array_equal(vc.view(torch.uint8).cpu().numpy().reshape(-1), vc_h)
    n = 0
    ids = w.decode_ids()
    if len(ids):
        ids, qq, bt, cl = decode_inputs(w, qd)
        out = torch.empty_like(qq)
        pkv.paged_attention_decode(out, qq, kc, vc, bt, cl, w.scale,
                                   max_context_len=int(w.context_lens[ids].max()), k_scale=ks,
                                   v_scale=vs, partition_size=partition_size, device_errors=err)
        qsl = workloads.query_start_loc(w.q_lens)
        qh = np.ascontiguousarray(q[qsl[ids]])
        ref = oracle.paged_attention_decode(qh, kc_h, vc_h, w.block_tables[ids],
                                            w.context_lens[ids], w.num_kv_heads, w.head_dim, 16,
                                            w.num_blocks, w.scale, w.q_dtype, w.kv_dtype, ks, vs)
        check_close(out.float().cpu().numpy(), ref, tol(w), f"{w.name} decode")
        n += ref.size
    ids = w.prefill_ids()
    if len(ids):
        ids, qq, bt, cl, qsl_d = prefill_inputs(w, qd)
        out = torch.empty_like(qq)
        pkv.paged_attention_prefill_chunk(out, qq, kc, vc, bt, cl, qsl_d, w.scale,
                                          max_q_len=int(w.q_lens[ids].max()),
                                          max_context_len=int(w.context_lens[ids].max()),
                                          k_scale=ks, v_scale=vs, device_errors=err)
        qsl = workloads.query_start_loc(w.q_lens)
        rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in ids])
        ref = oracle.paged_attention_prefill(np.ascontiguousarray(q[rows]), kc_h, vc_h,
                                             w.block_tables[ids], w.context_lens[ids],
                                             workloads.query_start_loc(w.q_lens[ids]),
                                             w.num_kv_heads, w.head_dim, 16, w.num_blocks,
                                             w.scale, w.q_dtype, w.kv_dtype, ks, vs)
        check_close(out.float().cpu().numpy(), ref, tol(w), f"{w.name} prefill")
        n += ref.size
    assert pkv.check_errors(err) == 0
    return n


@pytest.mark.parametrize("seed", range(5))
def test_tiny_config(seed):
    assert run_case(workloads.tiny(seed)) > 0


@pytest.mark.parametrize("src,cache", [(F16, F16), (BF16, BF16), (BF16, E4M3), (F16, E4M3)])
@pytest.mark.parametrize("D", [64, 128])
def test_reshape_and_cache_random_slots_bit_exact(src, cache, D):
    r = workloads.rng(500 + 10 * src + cache + D)
    nb, hkv, T = 40, 3, 200
    slots = r.choice(nb * 16, size=T, replace=False).astype(np.int64)
    slots[r.choice(T, size=7, replace=False)] = -1  # padding entries are skipped
    k = workloads.normal_bits(int(r.integers(1 << 30)), (T, hkv, D), src)
    v = workloads.normal_bits(int(r.integers(1 << 30)), (T, hkv, D), src)
    eb = 1 if cache == E4M3 else 2
    ks = vs = 1.0
    if cache == E4M3:
        # a scale small enough that part of the values saturate at +-448
        ks, vs = fp8_scale(k, src) / 3.0, fp8_scale(v, src)
    kh = np.full(nb * hkv * 16 * D * eb, 0x5A, np.uint8)
    vh = kh.copy()
    oracle.reshape_and_cache(k, v, kh, vh, slots, nb, 16, src, cache, ks, vs)
    kd = torch.full((nb, hkv, 16, D * eb), 0x5A, dtype=torch.uint8, device="cuda")
    vd = kd.clone()
    if cache != E4M3:
        kd, vd = kd.view(torch.int16).view(pkv_dtype(cache)), vd.view(torch.int16).view(pkv_dtype(cache))
    pkv.reshape_and_cache(bits_to_dev(k, src), bits_to_dev(v, src), kd, vd,
                          torch.from_numpy(slots).cuda(), ks, vs)
    assert np.array_equal(kd.view(torch.uint8).cpu().numpy().reshape(-1), kh)
    assert np.array_equal(vd.view(torch.uint8).cpu().numpy().reshape(-1), vh)


def pkv_dtype(code):
    return {F16: torch.float16, BF16: torch.bfloat16}[code]


@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("kv", [BF16, E4M3])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_block_boundaries(g, kv, D):
    ctx = [1, 15, 16, 17, 31, 32, 33, 100, 511, 512, 513, 1500]
    w = workloads.independent("edges", 1000 + g + D + kv, ctx, 2 * g, 2, D, BF16, kv)
    run_case(w)


@pytest.mark.parametrize("g", [2, 4, 8, 16])
@pytest.mark.parametrize("kv", [BF16, E4M3])
def test_decode_few_keys(g, kv):
    """Contexts of 2 to 40 tokens, next to long ones: rows that see a few keys,
    where weights rounded to the MMA input type alone would not meet the
    tolerance, in launches with and without partition merges."""
    ctx = list(range(2, 41)) + [1300]
    w = workloads.independent("few-keys", 1100 + g + kv, ctx, 2 * g, 2, 128, BF16, kv)
    run_case(w)
    w = workloads.independent("few-keys-1p", 1200 + g + kv, list(range(2, 41)), 2 * g, 2, 128,
                              BF16, kv)
    run_case(w)


@pytest.mark.parametrize("ps", [16, 64, 176, 512])
def test_decode_partition_sizes(ps):
    w = workloads.independent("parts", 2000 + ps, [1, 17, 300, 1024, 1777], 8, 2, 128, F16, F16)
    run_case(w, partition_size=ps)


def test_decode_empty_and_single_token_contexts():
    w = workloads.independent("empty", 31, [0, 1, 0, 2, 700], 4, 4, 64, BF16, BF16)
    run_case(w)


def test_decode_zero_contexts_single_pass():
    w = workloads.independent("empty2", 32, [0, 3, 0], 4, 2, 128, BF16, BF16)
    run_case(w)


@pytest.mark.parametrize("case", range(60))
def test_seeded_sweep(case):
    r = workloads.rng(7000 + case)
    S = int(r.integers(1, 7))
    hkv = int(r.choice([1, 2, 4]))
    g = int(r.choice([1, 2, 3, 4, 5, 6, 8, 16]))
    D = int(r.choice([64, 128]))
    qd = int(r.choice([F16, BF16]))
    kv = qd if r.random() < 0.6 else E4M3
    ctx = r.integers(0, 1300, size=S)
    q_lens = None
    if r.random() < 0.3:
        q_lens = [int(min(c, r.integers(1, 70))) if c > 0 else 0 for c in ctx]
        ctx = [max(int(c), ql) for c, ql in zip(ctx, q_lens)]
        if all(ql <= 1 for ql in q_lens):
            q_lens[0] = min(2, int(ctx[0])) if ctx[0] > 1 else q_lens[0]
    w = workloads.independent(f"sweep{case}", 7000 + case, ctx, hkv * g, hkv, D, qd, kv,
                              q_lens=q_lens)
    run_case(w, partition_size=int(r.choice([0, 32, 256])))


@pytest.mark.parametrize("g", [1, 4, 8])
def test_prefill_chunks(g):
    ctx = [40, 17, 64, 600, 700]
    qlen = [40, 5, 33, 512, 1]
    w = workloads.independent("prefill", 3000 + g, ctx, 2 * g, 2, 128, BF16, BF16, q_lens=qlen)
    run_case(w)


@pytest.mark.parametrize("g,qd", [(1, BF16), (2, F16), (4, BF16), (8, BF16), (16, F16)])
def test_prefill_chunks_e4m3_cache(g, qd):
    """Chunks over an E4M3 cache on the tensor-core prefill (8-bit MMAs over a
    query split into two E4M3 terms): partial last blocks, a chunk longer than
    one query tile, a single-token chunk, chunks from position 0."""
    ctx = [40, 17, 64, 600, 700, 1200, 33]
    qlen = [40, 5, 33, 512, 1, 300, 33]
    w = workloads.independent("prefill-e4m3", 3200 + g, ctx, 2 * g, 2, 128, qd, E4M3, q_lens=qlen)
    run_case(w)


@pytest.mark.parametrize("seed,g,dt", [(0, 4, BF16), (1, 8, F16), (2, 2, BF16), (3, 4, F16)])
def test_prefill_from_position_zero(seed, g, dt):
    """Whole prompts as chunks (no prior context): the first rows see one to a
    few dozen keys, where 16-bit softmax weights alone would not meet the
    tolerance; chunks shorter and longer than the recomputed rows, and one
    starting just inside them."""
    qlen = [5, 31, 32, 33, 200, 17]
    ctx = [5, 31, 32, 33, 200, 17 + 20]
    w = workloads.independent("prefill-from-0", 3100 + seed, ctx, 4 * g, 4, 128, dt, dt,
                              q_lens=qlen)
    run_case(w)


def test_mixed_small():
    w = workloads.mixed(seed=5, num_decode=6, num_prefill=2, chunk=96, prior=200)
    run_case(w)


def test_shared_prefix_small():
    w = workloads.gqa70b_shared(seed=6, num_seqs=10)
    run_case(w)


def test_device_checks_flag_bad_inputs():
    w = workloads.independent("bad", 41, [40, 50], 4, 2, 64, BF16, BF16)
    k, v, q = workloads.values_cpu(w)
    kc, vc = cache_tensors(w)
    err = errors_word()
    fill_device_cache(w, bits_to_dev(k, BF16), bits_to_dev(v, BF16), kc, vc, errors=err)
    assert pkv.check_errors(err) == 0
    qd = bits_to_dev(q, BF16)
    ids, qq, bt, cl = decode_inputs(w, qd)
    out = torch.empty_like(qq)
    bad = bt.clone()
    bad[1, 1] = w.num_blocks + 5
    pkv.paged_attention_decode(out, qq, kc, vc, bad, cl, w.scale, max_context_len=64,
                               device_errors=err)
    assert pkv.check_errors(err) & 0x1
    # a context longer than max_context_len is clamped and flagged
    pkv.paged_attention_decode(out, qq, kc, vc, bt, cl, w.scale, max_context_len=32,
                               partition_size=16, device_errors=err)
    assert pkv.check_errors(err) & 0x2
    # a slot beyond the pool is skipped and flagged
    slots = torch.tensor([0, w.num_blocks * 16 + 3], dtype=torch.int64, device="cuda")
    kk = bits_to_dev(k[:2], BF16)
    pkv.reshape_and_cache(kk, kk, kc, vc, slots, device_errors=err)
    assert pkv.check_errors(err) & 0x4
    assert pkv.check_errors(err) == 0


# ---- full-size workloads: every sequence against the oracle ------------------------------
def _workers(n):
    return max(1, min(n, os.cpu_count() or 1))


def _seq_bits(t, rows):
    """Source rows of one sequence as host uint16 bits."""
    return t.index_select(0, rows).cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _compact(w, c):
    """A one-sequence workload of c tokens on consecutive blocks 0.. (the
    oracle's result does not depend on the physical layout)."""
    nb = -(-c // 16)
    return workloads.Workload(
        name="sample", num_heads=w.num_heads, num_kv_heads=w.num_kv_heads,
        head_dim=w.head_dim, q_dtype=w.q_dtype, kv_dtype=w.kv_dtype, num_blocks=nb,
        context_lens=np.array([c], np.int32), q_lens=np.array([1], np.int32),
        block_tables=np.arange(nb, dtype=np.int32)[None], seq_rows=[np.arange(c)],
        num_src_rows=c, fill_rows=np.arange(c, dtype=np.int64),
        fill_slots=np.arange(c, dtype=np.int64), new_rows=np.zeros(0, np.int64),
        new_slots=np.zeros(0, np.int64), scale=w.scale, src_dtype=w.src_dtype)


def _sampled_oracle(w, k_src, v_src, q_all, sample, ks=1.0, vs=1.0):
    """Oracle output of the given decode sequences, each from a compact cache of
    its own source rows, one sequence per host thread (the oracle's C calls
    release the interpreter lock)."""
    qsl = workloads.query_start_loc(w.q_lens)

    def one(s):
        rows = torch.from_numpy(w.seq_rows[s]).to(k_src.device)
        kb, vb = _seq_bits(k_src, rows), _seq_bits(v_src, rows)
        sub = _compact(w, len(w.seq_rows[s]))
        kc_h, vc_h = host_cache(sub, kb, vb, ks, vs)
        qh = q_all[int(qsl[s]):int(qsl[s]) + 1].cpu().contiguous().view(torch.int16).numpy()
        return oracle.paged_attention_decode(
            qh.view(np.uint16), kc_h, vc_h, sub.block_tables, sub.context_lens, w.num_kv_heads,
            w.head_dim, 16, sub.num_blocks, w.scale, w.q_dtype, w.kv_dtype, ks, vs)[0]

    with ThreadPoolExecutor(_workers(len(sample))) as ex:
        return np.stack(list(ex.map(one, sample)))


def _full_size(w, ks_from_data=False):
    """Runs the workload's decode at full size and compares EVERY sequence with
    the oracle; returns the device state and the oracle's output."""
    dev = "cuda"
    k, v, q = workloads.values_device(w, dev)
    ks = vs = 1.0
    if ks_from_data:
        ks = float(np.float32(k.float().abs().max().item()) / np.float32(448.0))
        vs = float(np.float32(v.float().abs().max().item()) / np.float32(448.0))
    kc, vc = cache_tensors(w)
    err = errors_word()
    fill_device_cache(w, k, v, kc, vc, ks, vs, errors=err)
    ids, qq, bt, cl = decode_inputs(w, q)
    out = torch.empty_like(qq)
    pkv.paged_attention_decode(out, qq, kc, vc, bt, cl, w.scale,
                               max_context_len=int(w.context_lens[ids].max()), k_scale=ks,
                               v_scale=vs, device_errors=err)
    assert pkv.check_errors(err) == 0
    got = out.float().cpu().numpy()
    ref = _sampled_oracle(w, k, v, q, list(ids), ks, vs)
    check_close(got, ref, tol(w), w.name)
    return kc, vc, k, v, q, ks, vs, ref


def test_full_llama2_7b_every_sequence():
    _full_size(workloads.llama2_7b())


def test_full_gqa70b_shared_and_cascade_every_sequence():
    """The full 70B-GQA workload, every sequence, through plain decode and
    through the cascade entry point (shared prompts read once per group)."""
    w = workloads.gqa70b_shared()
    kc, vc, k, v, q, _, _, ref = _full_size(w)
    ids, qq, bt, cl = decode_inputs(w, q)
    gs, pre = w.cascade_groups()
    mx, mp = int(w.context_lens.max()), int(pre.max())
    err = errors_word()
    out = torch.empty_like(qq)
    pkv.paged_attention_decode_cascade(out, qq, kc, vc, bt, cl, torch.from_numpy(gs).cuda(),
                                       torch.from_numpy(pre).cuda(), w.scale, max_context_len=mx,
                                       max_prefix_len=mp, device_errors=err)
    assert pkv.check_errors(err) == 0
    check_close(out.float().cpu().numpy(), ref, tol(w), "cascade " + w.name)


def test_full_long_fp8_every_sequence():
    _full_size(workloads.long_fp8(), ks_from_data=True)


def test_full_mixed_every_row():
    """Mixed batch at full size: all 32 decode rows and all 4 chunks of 512
    queries against the oracle.  Each chunk is checked in slices of 64
    queries: a slice of a chunk is itself a chunk (same block table, context
    cut after its last query), so the slices run on separate host threads."""
    w = workloads.mixed()
    dev = "cuda"
    k, v, q = workloads.values_device(w, dev)
    kc, vc = cache_tensors(w)
    err = errors_word()
    fill_device_cache(w, k, v, kc, vc, errors=err)
    ids, qq, bt, cl = decode_inputs(w, q)
    out = torch.empty_like(qq)
    pkv.paged_attention_decode(out, qq, kc, vc, bt, cl, w.scale,
                               max_context_len=int(w.context_lens[ids].max()), device_errors=err)
    pids, pq, pbt, pcl, pqsl = prefill_inputs(w, q)
    pout = torch.empty_like(pq)
    pkv.paged_attention_prefill_chunk(pout, pq, kc, vc, pbt, pcl, pqsl, w.scale,
                                      max_q_len=512, max_context_len=2560, device_errors=err)
    assert pkv.check_errors(err) == 0
    ref = _sampled_oracle(w, k, v, q, list(ids))
    check_close(out.float().cpu().numpy(), ref, tol(w), "mixed decode rows")
    qsl = workloads.query_start_loc(w.q_lens)
    caches = {}
    for s in pids:
        rows = torch.from_numpy(w.seq_rows[s]).to(dev)
        sub = _compact(w, len(w.seq_rows[s]))
        caches[s] = (sub, host_cache(sub, _seq_bits(k, rows), _seq_bits(v, rows)))
    qh_all = q.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    step = 64

    def one(task):
        s, a = task
        sub, (kc_h, vc_h) = caches[s]
        c = int(sub.context_lens[0])
        qlen = int(w.q_lens[s])
        b = min(a + step, qlen)
        qh = np.ascontiguousarray(qh_all[int(qsl[s]) + a:int(qsl[s]) + b])
        return oracle.paged_attention_prefill(
            qh, kc_h, vc_h, sub.block_tables, np.array([c - qlen + b], np.int32),
            np.array([0, b - a], np.int32), w.num_kv_heads, w.head_dim, 16, sub.num_blocks,
            w.scale, BF16, BF16)

    tasks = [(s, a) for s in pids for a in range(0, int(w.q_lens[s]), step)]
    with ThreadPoolExecutor(_workers(len(tasks))) as ex:
        parts = list(ex.map(one, tasks))
    got = pout.float().cpu().numpy()
    base = {s: sum(int(w.q_lens[t]) for t in pids if t < s) for s in pids}
    for (s, a), r in zip(tasks, parts):
        check_close(got[base[s] + a:base[s] + a + len(r)], r, tol(w), f"mixed chunk {s} @{a}")


def test_full_mixed_cache_write_bit_exact():
    """The mixed step's cache write at full size (2,080 new tokens through its
    random slot mapping into the 8-head pool), compared byte for byte with the
    oracle's cache write over the whole K and V caches."""
    w = workloads.mixed()
    k, v, _ = workloads.values_device(w, "cuda")
    kc, vc = cache_tensors(w, sentinel=0x5A)
    err = errors_word()
    r = torch.from_numpy(w.new_rows).cuda()
    kn, vn = k.index_select(0, r).contiguous(), v.index_select(0, r).contiguous()
    assert kn.shape[0] == 2080
    pkv.reshape_and_cache(kn, vn, kc, vc, torch.from_numpy(w.new_slots).cuda(), device_errors=err)
    assert pkv.check_errors(err) == 0
    kc_h = np.full(cache_bytes(w), 0x5A, np.uint8)
    vc_h = np.full(cache_bytes(w), 0x5A, np.uint8)
    oracle.reshape_and_cache(_seq_bits(k, r), _seq_bits(v, r), kc_h, vc_h, w.new_slots,
                             w.num_blocks, 16, BF16, BF16)
    assert np.array_equal(kc.view(torch.uint8).cpu().numpy().reshape(-1), kc_h)
    assert np.array_equal(vc.view(torch.uint8).cpu().numpy().reshape(-1), vc_h)


def test_decode_many_sequences_chunked_launches():
    # more sequences than one tensor-core launch takes: the host splits them
    r = workloads.rng(91)
    ctx = r.integers(0, 700, size=1100)
    w = workloads.independent("many", 91, ctx, 8, 2, 128, BF16, BF16)
    run_case(w)


@pytest.mark.parametrize("g", [9, 12, 16])
def test_decode_wide_groups(g):
    w = workloads.independent("wide", 4000 + g, [1, 129, 700, 1600], g, 1, 128, F16, F16)
    run_case(w)
