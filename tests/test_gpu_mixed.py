"""Mixed batches in one call (pkv_paged_attention_mixed): decode rows first,
then prefill chunks.  Each part is compared with the oracle's decode and
prefill (|gpu - ref| <= 2e-3 + 1e-2 |ref|).  The fused kernel runs the same
per-item arithmetic as the separate decode and prefill kernels, so at the full
mixed-batch size its output must equal theirs bit for bit, whatever the split
of CTAs between the two kinds of work."""
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


def device_inputs(w, with_host=True):
    k, v, q = workloads.values_cpu(w)
    kc_h = vc_h = None
    if with_host:
        kc_h, vc_h = host_cache(w, k, v)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc, vc = cache_tensors(w)
    fill_device_cache(w, bits_to_dev(k, w.src_dtype), bits_to_dev(v, w.src_dtype), kc, vc,
                      errors=err)
    qd = bits_to_dev(q, w.q_dtype).contiguous()
    bt = torch.from_numpy(np.ascontiguousarray(w.block_tables)).cuda()
    cl = torch.from_numpy(np.ascontiguousarray(w.context_lens)).cuda()
    qsl = torch.from_numpy(workloads.query_start_loc(w.q_lens)).cuda()
    return q, kc_h, vc_h, qd, kc, vc, bt, cl, qsl, err


def run_mixed(w, nd, prefill_ctas=0):
    """The first nd sequences are decode rows (one query each), the rest chunks."""
    assert (w.q_lens[:nd] == 1).all()
    q, kc_h, vc_h, qd, kc, vc, bt, cl, qsl, err = device_inputs(w)
    out = torch.full_like(qd, float("nan"))
    pkv.paged_attention_mixed(out, qd, kc, vc, bt, cl, qsl, nd, w.scale,
                              prefill_ctas=prefill_ctas, device_errors=err)
    assert pkv.check_errors(err) == 0
    got = out.float().cpu().numpy()
    if nd:
        ref = oracle.paged_attention_decode(np.ascontiguousarray(q[:nd]), kc_h, vc_h,
                                            w.block_tables[:nd], w.context_lens[:nd],
                                            w.num_kv_heads, w.head_dim, 16, w.num_blocks,
                                            w.scale, w.q_dtype, w.kv_dtype)
        check_close(got[:nd], ref, tol(w), f"{w.name} decode rows")
    if nd < w.num_seqs:
        qsl_h = workloads.query_start_loc(w.q_lens)
        ref = oracle.paged_attention_prefill(np.ascontiguousarray(q[nd:]), kc_h, vc_h,
                                             w.block_tables[nd:], w.context_lens[nd:],
                                             qsl_h[nd:] - nd, w.num_kv_heads, w.head_dim, 16,
                                             w.num_blocks, w.scale, w.q_dtype, w.kv_dtype)
        check_close(got[nd:], ref, tol(w), f"{w.name} chunk rows")


def batch(seed, dctx, chunks, H, Hkv, dt=BF16):
    """Decode rows with contexts dctx, then chunks (q_len, prior); returns the
    workload and the number of decode rows."""
    ctx = list(dctx) + [a + b for a, b in chunks]
    q_lens = [1] * len(dctx) + [a for a, _ in chunks]
    return workloads.independent("mixed", seed, ctx, H, Hkv, 128, dt, dt, q_lens=q_lens), len(dctx)


@pytest.mark.parametrize("g,dt", [(4, BF16), (8, F16), (2, BF16)])
def test_mixed_small(g, dt):
    # decode contexts around block and partition edges; chunks with and without
    # prior context, one shorter than a query tile, one spanning several
    w = batch(40 + g, [1, 16, 17, 511, 512, 513, 2000, 3001], [(100, 300), (37, 0), (256, 1024),
                                                               (1, 77)], 4 * g, 4, dt)
    run_mixed(*w)


@pytest.mark.parametrize("ctas", [1, 7, 151])
def test_mixed_forced_splits(ctas):
    w = batch(50, [700, 33, 4096, 5], [(130, 20), (64, 900)], 32, 8)
    run_mixed(*w, prefill_ctas=ctas)


def test_mixed_unfused_shapes_and_degenerate_batches():
    # 16 query heads per KV head: the two separate launches
    run_mixed(*batch(60, [300, 17], [(50, 100)], 32, 2))
    # chunks only, decode rows only
    run_mixed(*batch(61, [], [(70, 10), (5, 0)], 16, 4))
    run_mixed(*batch(62, [40, 600], [], 16, 4))


def test_full_mixed_equals_separate_calls():
    """The mixed-batch workload (32 decode rows, 4 chunks of 512 over 2048
    prior tokens): fused output equals the separate decode and prefill calls'
    bit for bit, for the automatic split and forced ones."""
    w = workloads.mixed()
    nd = len(w.decode_ids())
    _, _, _, qd, kc, vc, bt, cl, qsl, err = device_inputs(w, with_host=False)
    ref = torch.empty_like(qd)
    mx = int(w.context_lens.max())
    pkv.paged_attention_decode(ref[:nd], qd[:nd].contiguous(), kc, vc, bt[:nd].contiguous(),
                               cl[:nd].contiguous(), w.scale, max_context_len=mx,
                               device_errors=err)
    pre = torch.empty_like(qd[nd:])
    pkv.paged_attention_prefill_chunk(pre, qd[nd:].contiguous(), kc, vc, bt[nd:].contiguous(),
                                      cl[nd:].contiguous(), (qsl[nd:] - nd).contiguous(),
                                      w.scale, max_q_len=512, max_context_len=mx,
                                      device_errors=err)
    ref[nd:] = pre
    for ctas in (0, 20, 76, 140):
        out = torch.full_like(qd, float("nan"))
        pkv.paged_attention_mixed(out, qd, kc, vc, bt, cl, qsl, nd, w.scale, max_q_len=512,
                                  max_context_len=mx, prefill_ctas=ctas, device_errors=err)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), ctas
    assert pkv.check_errors(err) == 0
