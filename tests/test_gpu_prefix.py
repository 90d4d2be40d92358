"""Prefix caching and copy-on-write end to end: the library's host block pool
(BlockPool) hands out the blocks, the library's kernels write and read them,
and the results are compared with the oracle's pool (oracle.CachePool), cache
writes, block copies and attention on the same operations.  Block copies are
compared byte for byte; attention within |gpu - ref| <= 2e-3 + 1e-2 |ref|."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_98_gb300 as pkv
import workloads
from _gpu import TD, bits_to_dev, check_close

pytestmark = pytest.mark.gpu
BF16, E4M3 = workloads.BF16, workloads.E4M3
BS, HKV, H, D = 16, 2, 8, 128
TOL = (2e-3, 1e-2)


@pytest.fixture(scope="module", autouse=True)
def _library():
    from paged_kv_cache_98_gb300 import _build
    _build.build()
    pkv.load()
    torch.cuda.init()


@pytest.mark.parametrize("dt", [BF16, E4M3])
def test_copy_blocks_bit_exact(dt):
    nb = 40
    elem = 1 if dt == E4M3 else 2
    r = np.random.default_rng(5)
    k0 = r.integers(0, 256, nb * HKV * BS * D * elem, dtype=np.uint8)
    v0 = r.integers(0, 256, nb * HKV * BS * D * elem, dtype=np.uint8)
    shape = (nb, HKV, BS, D)
    cdt = torch.uint8 if dt == E4M3 else TD[dt]
    kc = torch.from_numpy(k0.copy()).cuda().view(cdt).view(shape)
    vc = torch.from_numpy(v0.copy()).cuda().view(cdt).view(shape)
    # destinations distinct and never a source of the same call
    pairs = np.array([[3, 17], [0, 39], [25, 1], [38, 2], [7, 8]], np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(kc, vc, torch.from_numpy(pairs).cuda(), device_errors=err)
    oracle.copy_blocks(k0, v0, pairs, nb)
    assert pkv.check_errors(err) == 0
    assert np.array_equal(kc.view(torch.uint8).cpu().numpy().ravel(), k0)
    assert np.array_equal(vc.view(torch.uint8).cpu().numpy().ravel(), v0)
    bad = torch.tensor([[1, nb]], dtype=torch.int32, device="cuda")
    before = kc.view(torch.uint8).clone()
    pkv.copy_blocks(kc, vc, bad, device_errors=err)
    assert pkv.check_errors(err) & 1  # PKV_DEVERR_BLOCK_ID, nothing copied
    assert torch.equal(kc.view(torch.uint8), before)  # bytes: random bits include NaNs


class Both:
    """The library's pool and caches on the GPU, the oracle's on the host, fed the
    same operations."""

    def __init__(self, nb, seed):
        self.nb, self.seed = nb, seed
        self.lp, self.op = pkv.BlockPool(nb), oracle.CachePool(nb)
        shape = (nb, HKV, BS, D)
        self.kc = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
        self.vc = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
        self.kh = np.zeros(nb * HKV * BS * D * 2, np.uint8)
        self.vh = np.zeros_like(self.kh)
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def arrive(self, prompt):
        lr, orq = self.lp.request(), self.op.request()
        m = lr.match_prefix(prompt)
        assert orq.match(prompt) == m
        self.append((lr, orq), prompt[m:], m)
        return (lr, orq), m

    def append(self, req, ids, pos0):
        lr, orq = req
        sl, cl = lr.append(ids)
        so, co = orq.append(ids)
        assert np.array_equal(sl, so) and cl == co
        if cl is not None:  # copy the shared block before writing into the copy
            pkv.copy_blocks(self.kc, self.vc, torch.tensor([cl], dtype=torch.int32,
                                                          device="cuda"), device_errors=self.err)
            oracle.copy_blocks(self.kh, self.vh, [co], self.nb)
        k, v = workloads.token_kv(self.seed, ids, np.arange(pos0, pos0 + len(ids)), HKV, D, BF16)
        pkv.reshape_and_cache(bits_to_dev(k, BF16), bits_to_dev(v, BF16), self.kc, self.vc,
                              torch.from_numpy(sl).cuda(), device_errors=self.err)
        oracle.reshape_and_cache(k, v, self.kh, self.vh, so, self.nb, BS, BF16, BF16)
        assert np.array_equal(lr.block_table(), orq.table())

    def tables(self, reqs):
        mb = max(len(r[0].block_table()) for r in reqs)
        bt, cl = self.lp.block_tables([r[0] for r in reqs], mb)
        return bt, cl


def test_prefix_hit_prefill_equals_full_attention():
    """Request A computes a prompt and leaves; B shares its first 10 blocks,
    matches them, computes only its own 37 tokens, and attends over the reused
    blocks: equal to attention over B's whole context."""
    r = np.random.default_rng(11)
    both = Both(48, seed=21)
    pa = r.integers(0, 1024, 200)
    a, ma = both.arrive(pa)
    assert ma == 0
    a[0].free()
    a[1].free()
    pb = np.r_[pa[:160], r.integers(0, 1024, 37)]
    b, mb = both.arrive(pb)
    assert mb == 160
    bt, cl = both.tables([b])
    q = workloads.normal_bits(31, (37, H, D), BF16)
    qsl = np.array([0, 37], np.int32)
    out = torch.empty((37, H, D), dtype=torch.bfloat16, device="cuda")
    pkv.paged_attention_prefill_chunk(out, bits_to_dev(q, BF16), both.kc, both.vc,
                                      torch.from_numpy(bt).cuda(), torch.from_numpy(cl).cuda(),
                                      torch.from_numpy(qsl).cuda(), D ** -0.5, max_q_len=37,
                                      max_context_len=197, device_errors=both.err)
    assert pkv.check_errors(both.err) == 0
    ref = oracle.paged_attention_prefill(q, both.kh, both.vh, b[1].table()[None], [197], qsl,
                                         HKV, D, BS, both.nb, D ** -0.5, BF16, BF16)
    check_close(out.float().cpu().numpy(), ref, TOL, "prefix-hit prefill")
    # the reused blocks hold exactly A's K/V: the device cache equals the oracle's
    assert np.array_equal(both.kc.view(torch.uint8).cpu().numpy().ravel(), both.kh)


def test_forked_samples_copy_on_write_decode():
    """Three samples forked from one prompt with a partial last block each
    append tokens: the first two writers copy the shared block (device block
    copy), then every sample decodes over its own table."""
    r = np.random.default_rng(12)
    both = Both(64, seed=22)
    prompt = r.integers(0, 1024, 90)  # 5 full blocks + 10 tokens
    s0, _ = both.arrive(prompt)
    samples = [s0, (s0[0].fork(), s0[1].fork()), (s0[0].fork(), s0[1].fork())]
    n = len(prompt)
    for step in range(3):
        for s in samples:
            both.append(s, r.integers(0, 1024, 1), n)
        n += 1
    assert both.lp.num_free() == both.op.num_free() == 64 - 5 - 3
    bt, cl = both.tables(samples)
    q = workloads.normal_bits(32, (3, H, D), BF16)
    out = torch.empty((3, H, D), dtype=torch.bfloat16, device="cuda")
    pkv.paged_attention_decode(out, bits_to_dev(q, BF16), both.kc, both.vc,
                               torch.from_numpy(bt).cuda(), torch.from_numpy(cl).cuda(),
                               D ** -0.5, max_context_len=int(cl.max()), device_errors=both.err)
    assert pkv.check_errors(both.err) == 0
    ref = oracle.paged_attention_decode(q, both.kh, both.vh, bt, cl, HKV, D, BS, both.nb,
                                        D ** -0.5, BF16, BF16)
    check_close(out.float().cpu().numpy(), ref, TOL, "copy-on-write decode")
    assert np.array_equal(both.vc.view(torch.uint8).cpu().numpy().ravel(), both.vh)
