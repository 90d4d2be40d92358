"""Oracle block pool, block tables, slot mapping and byte model, pinned to the
pages' worked arithmetic (tests/golden/pages_worked_examples.txt) and to
closed-form invariants."""
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_worked_examples.txt")


def golden():
    vals = {}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (x.strip() for x in line.split("="))
            vals[k] = float(v) if "." in v else int(v)
    return vals


G = golden()


def test_kv_bytes_per_token_llama2_7b():
    # 4096 hidden = 32 heads x 128 per head, MHA, fp16.
    assert oracle.kv_bytes_per_token(32, 32, 128, 2) == G["kv_bytes_per_token_llama2_7b"]


def test_kv_bytes_per_token_gqa_models():
    assert oracle.kv_bytes_per_token(32, 8, 128, 2) == G["kv_bytes_per_token_llama3_8b"]
    assert oracle.kv_bytes_per_token(80, 8, 128, 2) == G["kv_bytes_per_token_llama3_70b"]
    # per layer, the figure every workload here reads per token and KV head group
    assert oracle.kv_bytes_per_token(1, 8, 128, 2) * 80 == G["kv_bytes_per_token_llama3_70b"]


def test_blocks_for_100_tokens_and_saving():
    bs = G["block_size"]
    n = oracle.blocks_for_tokens(100, bs)
    assert n == G["blocks_for_100_tokens"]
    half_mb = G["kv_bytes_per_token_llama2_7b"] / 2**20
    assert n * bs * half_mb == G["allocated_mb_for_100_tokens"]
    assert 2048 * half_mb == G["prealloc_mb_2048_tokens"]
    saving = 100.0 * (G["prealloc_mb_2048_tokens"] - n * bs * half_mb) / G["prealloc_mb_2048_tokens"]
    assert round(saving, 1) == G["saving_percent_100_tokens"]


@pytest.mark.parametrize("n", [0, 1, 15, 16, 17, 31, 32, 33, 100, 1000])
def test_pool_append_matches_ceil(n):
    pool = oracle.Pool(200)
    s = oracle.Seq(pool)
    s.append(n)
    assert s.num_tokens == n
    assert len(s.table()) == -(-n // 16)
    assert pool.num_free() == 200 - len(s.table())
    s.free()
    assert pool.num_free() == 200


def test_identity_pool_gives_consecutive_slots():
    # With blocks handed out 0, 1, 2, ... a single sequence's tokens occupy
    # consecutive slots 0..n-1.
    pool = oracle.Pool(10)
    s = oracle.Seq(pool)
    slots = s.append(150)
    assert np.array_equal(slots, np.arange(150))
    assert [s.slot(p) for p in range(150)] == list(range(150))
    assert s.slot(150) == -1


def test_slots_scattered_pool_invariants():
    r = workloads.rng(5)
    order = r.permutation(64).astype(np.int32)
    pool = oracle.Pool(64, order)
    seqs = [oracle.Seq(pool) for _ in range(3)]
    all_slots = []
    # interleaved appends: blocks of different sequences alternate in the pool
    for step in range(5):
        for i, s in enumerate(seqs):
            all_slots.append(s.append(7 + 3 * i + step))
    all_slots = np.concatenate(all_slots)
    assert len(np.unique(all_slots)) == len(all_slots)
    for s in seqs:
        t = s.table()
        for p in range(s.num_tokens):
            sl = s.slot(p)
            assert sl // 16 == t[p // 16] and sl % 16 == p % 16
    # blocks come out of the pool in the free-list order
    used = set()
    for s in seqs:
        used.update(s.table().tolist())
    assert used == set(order[:len(used)].tolist())


def test_parallel_sampling_copy_on_write_worked_example():
    # A prompt filling 5 blocks and part of a 6th; three parallel samples
    # share it by reference; each sample then generates one token.
    pool = oracle.Pool(64)
    base = oracle.Seq(pool)
    base.append(5 * 16 + 7)
    samples = [base, base.fork(), base.fork()]
    prompt_blocks = base.table().tolist()
    assert len(prompt_blocks) == 6
    assert all(pool.ref_cnt(b) == G["parallel_sampling_ref_cnt"] for b in prompt_blocks)
    for s in samples:
        s.append(1)
    tables = [s.table().tolist() for s in samples]
    shared = set(tables[0][:5])
    assert all(set(t[:5]) == shared for t in tables)
    assert all(pool.ref_cnt(b) == 3 for b in shared)
    last = {t[5] for t in tables}
    assert len(last) == G["parallel_sampling_blocks_private"]
    in_use = 64 - pool.num_free()
    assert len(shared) == G["parallel_sampling_blocks_shared"]
    assert in_use == G["parallel_sampling_blocks_paged"]
    copied = 3 * len(prompt_blocks)
    assert copied == G["parallel_sampling_blocks_copied"]
    assert int(100 * (1 - in_use / copied)) == G["parallel_sampling_saving_percent"]
    for s in samples:
        s.free()
    assert pool.num_free() == 64
    assert all(pool.ref_cnt(b) == 0 for b in range(64))


def test_copy_on_write_copies_block_bytes():
    nb, hkv, d = 16, 2, 8
    block_bytes = hkv * 16 * d * 2
    r = workloads.rng(9)
    kc = r.integers(0, 256, size=nb * block_bytes, dtype=np.uint8)
    vc = r.integers(0, 256, size=nb * block_bytes, dtype=np.uint8)
    pool = oracle.Pool(nb)
    a = oracle.Seq(pool)
    a.append(20, (kc, vc, block_bytes))
    b = a.fork()
    old = a.table()[1]
    kb = kc.copy()
    b.append(1, (kc, vc, block_bytes))
    new = b.table()[1]
    assert new != old and pool.ref_cnt(old) == 1 and pool.ref_cnt(new) == 1
    assert np.array_equal(kc[new * block_bytes:(new + 1) * block_bytes],
                          kb[old * block_bytes:(old + 1) * block_bytes])
    assert np.array_equal(vc[new * block_bytes:(new + 1) * block_bytes],
                          vc[old * block_bytes:(old + 1) * block_bytes])
    # the full first block stays shared
    assert a.table()[0] == b.table()[0] and pool.ref_cnt(a.table()[0]) == 2


def test_free_releases_tail_first():
    pool = oracle.Pool(8)
    s = oracle.Seq(pool)
    s.append(40)
    t = s.table().tolist()
    s.free()
    # the free list is popped from its end: the blocks released last (the
    # prefix) come out first, in table order
    assert [pool.alloc() for _ in range(3)] == t


def test_pool_exhaustion_and_double_free():
    pool = oracle.Pool(2)
    s = oracle.Seq(pool)
    s.append(32)
    with pytest.raises(oracle.OracleError):
        s.append(1)
    assert pool.alloc() == -1
    b = s.table()[0]
    assert pool.decref(b) == 0
    assert pool.decref(b) == -1  # already free
    assert pool.incref(b) == -1  # a free block cannot gain a reference


def test_workload_tables_match_pool_construction():
    # The synthetic generator lays blocks out as a pool handing out the same
    # permutation would.
    w = workloads.independent("t", 3, [5, 40, 16, 33], 2, 2, 8, workloads.F16, workloads.F16)
    order = workloads.rng(3).permutation(w.num_blocks).astype(np.int32)
    pool = oracle.Pool(w.num_blocks, order)
    for s in range(w.num_seqs):
        seq = oracle.Seq(pool)
        slots = seq.append(int(w.context_lens[s]))
        nb = len(seq.table())
        assert np.array_equal(seq.table(), w.block_tables[s, :nb])
        # the step's new token is the last position
        assert slots[-1] == w.new_slots[s]


def test_shared_prefix_workload_structure():
    prompts, tails = [37, 16, 100], [[3, 20, 1], [5, 5], [1]]
    w = workloads.shared_prefix("s", 4, prompts, tails, 2, 1, 8, workloads.BF16, workloads.BF16)
    used_private = []
    for P, g in zip(prompts, w.shared_groups):
        full = P // 16
        first = g[0]
        for s in g:
            assert w.context_lens[s] == P + tails[prompts.index(P)][g.index(s)]
            # same prompt tokens, same physical prompt blocks
            assert np.array_equal(w.seq_rows[s][:P], w.seq_rows[first][:P])
            assert np.array_equal(w.block_tables[s, :full], w.block_tables[first, :full])
            nb = -(-int(w.context_lens[s]) // 16)
            used_private.extend(w.block_tables[s, full:nb].tolist())
    # private blocks (including the copied partial prompt block) are per sample
    assert len(set(used_private)) == len(used_private)
    # all cache writes land on distinct slots
    slots = np.concatenate([w.fill_slots, w.new_slots])
    assert len(np.unique(slots)) == len(slots)
