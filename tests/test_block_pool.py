"""The library's host block pool (pkv_block_pool_* / pkv_request_*) against the
oracle's prefix-caching pool: on the same operations both must hand out the
same blocks, slots and copy-on-write pairs, keep the same free-queue order and
reference counts, and cache the same blocks.  Plus the worked example of
"第34讲 … vLLM 生产级系统架构全景剖析与四重加速引擎" §2.2 run on the library
itself, argument checks, and the batch block-table builder."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_98_gb300 as pkv
from paged_kv_cache_98_gb300 import _build

BS = 16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    pkv.load()


def same_state(lp, op, nb):
    assert np.array_equal(lp.queue(), op.queue())
    assert lp.num_free() == op.num_free() and lp.num_cached() == op.num_cached()
    for b in range(nb):
        assert lp.ref_cnt(b) == op.ref_cnt(b)
        assert lp.is_cached(b) == op.is_cached(b)


def test_page_prefix_example_on_library():
    r = np.random.default_rng(1)
    kb = r.integers(0, 32000, 62 * BS)
    p = pkv.BlockPool(256)
    u1 = np.r_[kb, r.integers(0, 32000, 15)]
    u2 = np.r_[kb, r.integers(0, 32000, 12)]
    a = p.request()
    assert a.match_prefix(u1) == 0
    a.append(u1)
    b = p.request()
    m = b.match_prefix(u2)
    assert len(u2) - m == 12
    b.append(u2[m:])
    ta, tb = a.block_table(), b.block_table()
    assert np.array_equal(tb[:62], ta[:62]) and np.array_equal(ta[:62], np.arange(62))
    assert (ta[62] + 1, tb[62] + 1) == (63, 64)  # the figure's blocks #63 and #64
    assert all(p.ref_cnt(i) == 2 for i in range(62))
    p.close()


@pytest.mark.parametrize("seed", range(6))
def test_matches_oracle_on_random_traces(seed):
    """Arrivals drawn from a few shared prompts (prefix matching), decode appends,
    forks and frees on a pool small enough to evict; every result compared."""
    r = np.random.default_rng(100 + seed)
    nb = int(r.integers(40, 200))
    lp, op = pkv.BlockPool(nb), oracle.CachePool(nb)
    prompts = [r.integers(0, 300, int(r.integers(10, 180))) for _ in range(6)]
    live = []  # (library request, oracle request)
    stats = {"hits": 0, "cow": 0, "full": 0, "evict": 0}
    for step in range(400):
        x = r.random()
        if x < 0.3 or not live:
            base = prompts[int(r.integers(len(prompts)))]
            toks = np.r_[base[:int(r.integers(1, len(base) + 1))],
                         r.integers(0, 300, int(r.integers(0, 30)))]
            if len(toks) == 0:
                continue
            lr, orq = lp.request(), op.request()
            ml, mo = lr.match_prefix(toks), orq.match(toks)
            assert ml == mo
            stats["hits"] += ml
            cached_before = lp.num_cached()
            try:
                sl, cl = lr.append(toks[ml:])
            except pkv.PagedKVError as e:
                assert e.status == -7
                with pytest.raises(oracle.OracleError):
                    orq.append(toks[mo:])
                stats["full"] += 1
                lr.free()
                orq.free()
                continue
            so, co = orq.append(toks[mo:])
            assert np.array_equal(sl, so) and cl == co
            stats["evict"] += lp.num_cached() < cached_before
            live.append((lr, orq))
        elif x < 0.65:
            i = int(r.integers(len(live)))
            lr, orq = live[i]
            ids = r.integers(0, 300, int(r.integers(1, 24)))
            try:
                sl, cl = lr.append(ids)
            except pkv.PagedKVError:
                with pytest.raises(oracle.OracleError):
                    orq.append(ids)
                stats["full"] += 1
                continue
            so, co = orq.append(ids)
            assert np.array_equal(sl, so) and cl == co
            stats["cow"] += cl is not None
        elif x < 0.75:
            lr, orq = live[int(r.integers(len(live)))]
            live.append((lr.fork(), orq.fork()))
        else:
            lr, orq = live.pop(int(r.integers(len(live))))
            lr.free()
            orq.free()
        for lr, orq in live:
            assert np.array_equal(lr.block_table(), orq.table())
            assert lr.num_tokens == orq.num_tokens
        same_state(lp, op, nb)
    assert min(stats.values()) > 0  # hits, copies on write, exhaustion, evictions
    lp.close()


def test_batch_block_tables():
    p = pkv.BlockPool(64)
    a, b = p.request(), p.request()
    a.append(np.arange(40))
    b.append(np.arange(3))
    bt, cl = p.block_tables([a, b], 5)
    assert cl.tolist() == [40, 3]
    assert bt[0, :3].tolist() == a.block_table().tolist() and bt[0, 3:].tolist() == [0, 0]
    assert bt[1, 0] == b.block_table()[0]
    with pytest.raises(pkv.PagedKVError):
        p.block_tables([a], 2)  # a holds 3 blocks
    p.close()


def test_argument_checks():
    lib = pkv.load()
    import ctypes
    h = ctypes.c_void_p()
    assert lib.pkv_block_pool_create(-1, 16, ctypes.byref(h)) == -1 and not h.value
    assert lib.pkv_block_pool_create(4, 0, ctypes.byref(h)) == -1
    assert lib.pkv_block_pool_num_free(None) == -1
    p = pkv.BlockPool(4)
    a = p.request()
    a.append([1, 2, 3])
    with pytest.raises(pkv.PagedKVError):
        a.match_prefix(np.arange(40))  # not an empty request
    assert p.ref_cnt(4) == -1 and p.ref_cnt(-1) == -1
    with pytest.raises(pkv.PagedKVError) as e:
        a.append(np.arange(4 * BS))  # 4 more blocks, 3 free
    assert e.value.status == -7 and a.num_tokens == 3 and p.num_free() == 3
    p.close()
