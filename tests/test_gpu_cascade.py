"""Cascade (shared-prefix) decode vs the CPU oracle's plain decode.

The cascade reads each group's shared prompt blocks once and merges the
partial results with each sequence's own keys; its output must equal plain
attention over the whole context, so the oracle is the same decode
definition.  Tolerance as for decode: |gpu - ref| <= 2e-3 + 1e-2 |ref|.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_98_gb300 as pkv
import workloads
from _gpu import bits_to_dev, cache_tensors, check_close, decode_inputs, fill_device_cache, tol
from _util import host_cache

pytestmark = pytest.mark.gpu
F16, BF16 = workloads.F16, workloads.BF16


@pytest.fixture(scope="module", autouse=True)
def _library():
    from paged_kv_cache_98_gb300 import _build
    _build.build()
    pkv.load()
    torch.cuda.init()


def run_cascade(w, sentinel=0xFF, groups=None):
    """Runs the cascade decode of the workload's decode sequences and checks
    it against the oracle; returns the device error bits."""
    k, v, q = workloads.values_cpu(w)
    kc_h, vc_h = host_cache(w, k, v)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc, vc = cache_tensors(w, sentinel=sentinel)
    fill_device_cache(w, bits_to_dev(k, w.src_dtype), bits_to_dev(v, w.src_dtype), kc, vc,
                      errors=err)
    ids, qq, bt, cl = decode_inputs(w, bits_to_dev(q, w.q_dtype))
    gs, pre = w.cascade_groups() if groups is None else groups
    out = torch.empty_like(qq)
    pkv.paged_attention_decode_cascade(out, qq, kc, vc, bt, cl, torch.from_numpy(gs).cuda(),
                                       torch.from_numpy(pre).cuda(), w.scale, device_errors=err)
    bits = pkv.check_errors(err)
    qsl = workloads.query_start_loc(w.q_lens)
    ref = oracle.paged_attention_decode(np.ascontiguousarray(q[qsl[ids]]), kc_h, vc_h,
                                        w.block_tables[ids], w.context_lens[ids], w.num_kv_heads,
                                        w.head_dim, 16, w.num_blocks, w.scale, w.q_dtype,
                                        w.kv_dtype)
    if bits == 0:
        check_close(out.float().cpu().numpy(), ref, tol(w), f"{w.name} cascade")
    return bits


@pytest.mark.parametrize("g,dt", [(8, BF16), (4, F16), (2, BF16), (16, BF16)])
def test_cascade_shared_groups(g, dt):
    # groups of 3, 1 and 2 samples; prompts with and without a partial block,
    # one shorter than a block, one spanning several 2048-key chunks
    prompts = [40, 100, 7, 300, 5000, 16]
    tails = [[1, 2, 3], [5], [16, 1], [200, 3, 64], [9, 130], [1, 1]]
    w = workloads.shared_prefix("cascade", 11, prompts, tails, 2 * g, 2, 128, dt, dt)
    gs, pre = w.cascade_groups()
    assert pre.max() >= 4096  # the long prompt's prefix spans several chunks
    assert run_cascade(w) == 0


def test_cascade_gqa70b_shape():
    """The 70B-GQA shape (64 / 8 heads, groups of 3 with lognormal prompts),
    fewer sequences so the oracle runs in seconds."""
    w = workloads.gqa70b_shared(seed=5, num_seqs=24)
    assert run_cascade(w) == 0


def test_cascade_without_sharing_equals_decode():
    """Independent sequences: one group with no prefix, i.e. plain decode."""
    w = workloads.independent("cascade-indep", 12, [1, 17, 512, 513, 2000], 8, 2, 128, BF16,
                              BF16)
    gs, pre = w.cascade_groups()
    assert len(gs) == 2 and pre.max() == 0
    assert run_cascade(w) == 0


def test_cascade_whole_context_shared():
    """A group whose members' whole contexts are shared blocks except the
    newest token (prefix = context rounded down to blocks)."""
    w = workloads.shared_prefix("cascade-full", 13, [64, 2048], [[1, 1], [1, 1, 1]], 16, 2,
                                128, BF16, BF16)
    assert run_cascade(w) == 0


def test_cascade_bad_prefix_is_flagged():
    """A prefix that is not whole blocks is cut back and flagged (no fault)."""
    w = workloads.shared_prefix("cascade-bad", 14, [100], [[2, 3]], 8, 2, 128, BF16, BF16)
    gs, pre = w.cascade_groups()
    pre = pre.copy()
    pre[:] = 97  # not a multiple of 16
    bits = run_cascade(w, groups=(gs, pre))
    assert bits & 2  # PKV_DEVERR_CONTEXT


def test_cascade_unsupported_shapes():
    w = workloads.shared_prefix("cascade-fp8", 15, [64], [[1, 2]], 8, 2, 128, BF16,
                                workloads.E4M3)
    k, v, q = workloads.values_cpu(w)
    kc, vc = cache_tensors(w)
    ids, qq, bt, cl = decode_inputs(w, bits_to_dev(q, w.q_dtype))
    gs, pre = w.cascade_groups()
    out = torch.empty_like(qq)
    with pytest.raises(pkv.PagedKVError):
        pkv.paged_attention_decode_cascade(out, qq, kc, vc, bt, cl, torch.from_numpy(gs).cuda(),
                                           torch.from_numpy(pre).cuda(), w.scale)
