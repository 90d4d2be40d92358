"""Oracle prefix-caching pool (oracle.CachePool), pinned to the worked example
of "第34讲 … vLLM 生产级系统架构全景剖析与四重加速引擎" §2.2 (tests/golden), to the
queue discipline §1.2 and §2.3 state (tail-first release, ref_cnt 0 blocks
appended at the tail, allocation from the head), and to content invariants
checked through a simulated cache: every slot a request reads holds the token
that request has at that position."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_worked_examples.txt")
BS = 16


def golden():
    vals = {}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (x.strip() for x in line.split("="))
                vals[k] = float(v) if "." in v else int(v)
    return vals


G = golden()


def test_page_prefix_example():
    """§2.2 figure: a knowledge-base prefix on blocks #1-#62 shared by two users
    (ref_cnt 2); each user's question in a private block (#63, #64), and only the
    question's tokens are computed.  The page's block numbers count from 1; a fresh
    pool hands out block ids 0, 1, 2, ..."""
    r = np.random.default_rng(1)
    nshared = G["prefix_shared_blocks"]
    kb = r.integers(0, 32000, nshared * BS)
    p = oracle.CachePool(256)
    u1 = np.r_[kb, r.integers(0, 32000, G["prefix_user1_new_tokens"])]
    u2 = np.r_[kb, r.integers(0, 32000, G["prefix_user2_new_tokens"])]
    a = p.request()
    assert a.match(u1) == 0  # nothing cached yet
    a.append(u1)
    b = p.request()
    hit = b.match(u2)
    assert len(u2) - hit == G["prefix_user2_new_tokens"]
    b.append(u2[hit:])
    ta, tb = a.table(), b.table()
    assert np.array_equal(ta[:nshared], np.arange(nshared))
    assert np.array_equal(tb[:nshared], ta[:nshared])
    assert ta[nshared] + 1 == G["prefix_user1_block"]
    assert tb[nshared] + 1 == G["prefix_user2_block"]
    assert all(p.ref_cnt(i) == G["prefix_shared_ref_cnt"] for i in range(nshared))
    assert p.ref_cnt(ta[nshared]) == 1 and p.ref_cnt(tb[nshared]) == 1


def test_release_is_tail_first_to_queue_tail():
    """§1.2: a finished request frees its blocks in reverse order; §2.3: blocks at
    ref_cnt 0 join the free queue's tail and stay cached."""
    p = oracle.CachePool(10)
    a = p.request()
    a.append(np.arange(3 * BS + 5))  # 3 full blocks + 1 partial
    t = a.table()
    before = p.queue()
    a.free()
    assert np.array_equal(p.queue(), np.r_[before, t[::-1]])
    assert p.num_cached() == 3
    assert [p.is_cached(int(i)) for i in t] == [True, True, True, False]


def test_allocation_takes_the_head_and_evicts():
    """§2.3: when blocks run short, the head of the free queue (least recently
    released) is reused first and its cached prefix stops matching."""
    p = oracle.CachePool(6)
    a = p.request()
    toks = np.arange(4 * BS) + 100
    a.append(toks)
    a.free()  # queue: 4 5 | a3 a2 a1 a0
    ta = [0, 1, 2, 3]
    x = p.request()
    q0 = p.queue()
    x.append(np.arange(3 * BS) + 5000)  # takes 4, 5 and then evicts a3
    assert np.array_equal(x.table(), q0[:3])
    assert x.table()[2] == ta[3]
    assert p.num_cached() == 6  # a0-a2 still cached, x's three blocks registered
    b = p.request()
    assert b.match(np.r_[toks, 1]) == 3 * BS  # a0-a2 hit, a3 was evicted


def test_hit_takes_block_from_middle_of_queue():
    """§1.2: a prefix hit revives a cached free block wherever it sits in the
    queue; it is then in use and no allocation can take it."""
    p = oracle.CachePool(8)
    a = p.request()
    toks = np.arange(2 * BS) + 7
    a.append(toks)
    a.free()  # queue: 2..7, a1, a0
    b = p.request()
    assert b.match(np.r_[toks[:BS], 9, 9]) == BS  # only a0's prefix
    assert 0 not in p.queue() and p.ref_cnt(0) == 1
    c = p.request()
    c.append(np.arange(7 * BS) + 900)  # everything else: 2..7 and a1
    assert sorted(c.table().tolist()) == [1, 2, 3, 4, 5, 6, 7]
    assert p.num_free() == 0 and p.ref_cnt(0) == 1


def test_whole_prompt_cached_leaves_last_block_to_compute():
    """A prompt whose every block is cached still computes its last block (the
    step needs at least one query); the recomputed block duplicates a cached
    prefix and stays unregistered."""
    p = oracle.CachePool(16)
    toks = np.arange(4 * BS) + 3
    a = p.request()
    a.append(toks)
    assert p.num_cached() == 4
    b = p.request()
    assert b.match(toks) == 3 * BS
    _, cow = b.append(toks[3 * BS:])
    assert cow is None
    assert p.num_cached() == 4 and not p.is_cached(int(b.table()[3]))
    assert np.array_equal(b.table()[:3], a.table()[:3])
    c = p.request()
    assert c.match(np.r_[toks, 1]) == 4 * BS  # the first copy serves the hit
    assert np.array_equal(c.table(), a.table())


def test_block_matches_only_under_its_own_prefix():
    """A cached block stands for its whole prefix: the same 16 tokens after a
    different first block are no hit, and a hit stops at the first miss."""
    p = oracle.CachePool(16)
    x, y, z = (np.full(BS, v) for v in (1, 2, 3))
    a = p.request()
    a.append(np.r_[x, y, z, 0])
    b = p.request()
    assert b.match(np.r_[z, y, z, 0]) == 0
    c = p.request()
    assert c.match(np.r_[x, z, z, 0]) == BS
    d = p.request()
    assert d.match(np.r_[x, y, z, 0]) == 3 * BS


def test_exhaustion_changes_nothing():
    p = oracle.CachePool(3)
    a = p.request()
    a.append(np.arange(BS + 3))
    q, t = p.queue(), a.table()
    with pytest.raises(oracle.OracleError):
        a.append(np.arange(3 * BS))  # needs 3 new blocks, 1 free
    assert np.array_equal(p.queue(), q) and np.array_equal(a.table(), t)
    assert a.num_tokens == BS + 3


def test_fork_copy_on_write_counts():
    """openeuler notes "机制 2：写时复制": three samples of a 6-block prompt whose 6th
    block is partial, one new token each: 5 shared + 3 private = 8 blocks, the
    shared ones at ref_cnt 3."""
    p = oracle.CachePool(32)
    a = p.request()
    a.append(np.arange(5 * BS + 4))
    b, c = a.fork(), a.fork()
    cows = [s.append([1000 + i])[1] for i, s in enumerate((a, b, c))]
    assert cows[0] is not None and cows[1] is not None and cows[2] is None
    used = {int(x) for s in (a, b, c) for x in s.table()}
    assert len(used) == G["parallel_sampling_blocks_paged"]
    assert all(p.ref_cnt(int(x)) == G["parallel_sampling_ref_cnt"] for x in a.table()[:5])
    assert p.num_free() == 32 - 8


class SimCache:
    """Token ids written to slots, standing in for K/V: a request reading its
    blocks must find its own tokens there."""

    def __init__(self, num_blocks):
        self.slot = np.full(num_blocks * BS, -1, np.int64)

    def write(self, slots, ids):
        self.slot[slots] = ids

    def copy_block(self, src, dst):
        self.slot[dst * BS:(dst + 1) * BS] = self.slot[src * BS:(src + 1) * BS]

    def check(self, req, tokens):
        t = req.table()
        assert len(t) == -(-len(tokens) // BS)
        pos = np.arange(len(tokens))
        assert np.array_equal(self.slot[t[pos // BS] * BS + pos % BS], tokens)


@pytest.mark.parametrize("seed", range(4))
def test_random_trace_content_and_queue_discipline(seed):
    """Random requests drawn from a few shared prompts: arrivals with prefix
    matching, decode appends, forks and frees.  After every operation the
    simulated cache holds each live request's tokens, blocks are either queued
    (ref 0) or referenced, allocations come from the queue's head in order, and
    releases go to its tail in reverse table order."""
    r = np.random.default_rng(seed)
    nb = 160
    p = oracle.CachePool(nb)
    sim = SimCache(nb)
    prompts = [r.integers(0, 500, int(r.integers(20, 200))) for _ in range(5)]
    live = []  # (req, tokens)
    hits = 0

    def append(req, toks, ids):
        q0 = p.queue()
        t0 = req.table()
        try:
            slots, cow = req.append(ids)
        except oracle.OracleError:
            assert np.array_equal(p.queue(), q0)
            return None
        t1 = req.table()
        new = [int(x) for x in t1[len(t0):]]
        taken = ([cow[1]] if cow else []) + new
        assert taken == [int(x) for x in q0[:len(taken)]]  # head first, in order
        if cow:
            sim.copy_block(*cow)
        sim.write(slots, ids)
        return np.r_[toks, ids]

    for _ in range(300):
        op = r.random()
        if op < 0.3 or not live:
            base = prompts[int(r.integers(len(prompts)))]
            toks = np.r_[base, r.integers(0, 500, int(r.integers(1, 40)))]
            req = p.request()
            m = req.match(toks)
            hits += m
            assert m % BS == 0 and m <= len(toks) - 1
            sim.check(req, toks[:m])
            got = append(req, toks[:m], toks[m:])
            if got is None:
                req.free()
                continue
            live.append((req, got))
        elif op < 0.7:
            i = int(r.integers(len(live)))
            req, toks = live[i]
            got = append(req, toks, r.integers(0, 500, int(r.integers(1, 20))))
            if got is not None:
                live[i] = (req, got)
        elif op < 0.8:
            req, toks = live[int(r.integers(len(live)))]
            live.append((req.fork(), toks))
        else:
            req, toks = live.pop(int(r.integers(len(live))))
            t = req.table()
            q0 = p.queue()
            refs = {int(x): p.ref_cnt(int(x)) for x in t}
            req.free()
            dropped = [int(x) for x in t[::-1] if refs[int(x)] == 1]
            assert np.array_equal(p.queue(), np.r_[q0, dropped].astype(np.int32))
        for req, toks in live:
            sim.check(req, toks)
        q = set(p.queue().tolist())
        assert all((p.ref_cnt(b) == 0) == (b in q) for b in range(nb))
    assert hits > 0


def test_copy_blocks_is_the_copy_of_copy_on_write():
    """oracle.copy_blocks reproduces the bytes that the block-table sequence's
    own copy-on-write (oracle.Seq.append with caches) writes, and touches no
    other block."""
    r = np.random.default_rng(3)
    nb, bb = 12, 8 * 16 * 64 * 2  # 8 KV heads x 16 rows x 64 dims x 2 bytes
    k0 = r.integers(0, 256, nb * bb, dtype=np.uint8)
    v0 = r.integers(0, 256, nb * bb, dtype=np.uint8)
    k1, v1 = k0.copy(), v0.copy()
    pool = oracle.Pool(nb)
    s = oracle.Seq(pool)
    s.append(2 * BS + 3, caches=(k1, v1, bb))
    c = s.fork()
    before = s.table().copy()
    c.append(1, caches=(k1, v1, bb))  # copies the shared partial block
    src, dst = int(before[-1]), int(c.table()[-1])
    assert src != dst
    k2, v2 = k0.copy(), v0.copy()
    oracle.copy_blocks(k2, v2, [[src, dst]], nb)
    assert np.array_equal(k2, k1) and np.array_equal(v2, v1)
    changed = np.flatnonzero((k2 != k0).reshape(nb, bb).any(axis=1))
    assert set(changed.tolist()) <= {dst}
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(k2, v2, [[0, nb]], nb)
