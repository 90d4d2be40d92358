"""The library's calls inside CUDA graphs: a step captured once (cache write,
attention, merge) and replayed after the inputs change in place must give the
same bytes as running the calls eagerly.  Capture fails loudly if a call
synchronises, allocates or reads device data on the host."""
import numpy as np
import pytest
import torch

import paged_kv_cache_98_gb300 as pkv
import workloads
from _gpu import bits_to_dev, cache_tensors, fill_device_cache

pytestmark = pytest.mark.gpu
BF16 = workloads.BF16


@pytest.fixture(scope="module", autouse=True)
def _library():
    from paged_kv_cache_98_gb300 import _build
    _build.build()
    pkv.load()
    torch.cuda.init()


def setup(w):
    k, v, q = workloads.values_cpu(w)
    kc, vc = cache_tensors(w)
    kd, vd = bits_to_dev(k, w.src_dtype), bits_to_dev(v, w.src_dtype)
    fill_device_cache(w, kd, vd, kc, vc, include_new=False)
    new = torch.from_numpy(w.new_rows).cuda()
    return dict(kc=kc, vc=vc, q=bits_to_dev(q, w.q_dtype).contiguous(),
                k_new=kd.index_select(0, new).contiguous(),
                v_new=vd.index_select(0, new).contiguous(),
                slots=torch.from_numpy(w.new_slots).cuda(),
                bt=torch.from_numpy(np.ascontiguousarray(w.block_tables)).cuda(),
                cl=torch.from_numpy(np.ascontiguousarray(w.context_lens)).cuda(),
                qsl=torch.from_numpy(workloads.query_start_loc(w.q_lens)).cuda(),
                err=torch.zeros(1, dtype=torch.int32, device="cuda"))


def replay_matches_eager(step, t, out):
    """Eager run, capture, replay; then new query values in place, replay and
    eager again.  Every output must match bit for bit."""
    step()
    torch.cuda.synchronize()
    ref = out.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    out.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    t["q"].copy_(torch.flip(t["q"], dims=[0]))  # new inputs, same buffers
    g.replay()
    torch.cuda.synchronize()
    got = out.clone()
    step()
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), out.view(torch.int16))
    assert not torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert pkv.check_errors(t["err"]) == 0


@pytest.mark.parametrize("H,Hkv", [(32, 8), (8, 8)])  # tensor-core and CUDA-core decode
def test_decode_step_in_a_graph(H, Hkv):
    w = workloads.independent("graph-decode", 90 + H, [1, 600, 2000, 4097], H, Hkv, 128, BF16,
                              BF16)
    t = setup(w)
    out = torch.empty_like(t["q"])
    ws = torch.empty(pkv.decode_workspace_size(4, H, 128, 4097) + 256, dtype=torch.uint8,
                     device="cuda")

    def step():
        pkv.reshape_and_cache(t["k_new"], t["v_new"], t["kc"], t["vc"], t["slots"],
                              device_errors=t["err"])
        pkv.paged_attention_decode(out, t["q"], t["kc"], t["vc"], t["bt"], t["cl"], w.scale,
                                   max_context_len=4097, workspace=ws, device_errors=t["err"])
    replay_matches_eager(step, t, out)


def test_cascade_decode_in_a_graph():
    w = workloads.shared_prefix("graph-cascade", 93, [300, 2500], [[1, 7, 30], [2, 90]], 32, 4,
                                128, BF16, BF16)
    t = setup(w)
    gs, pre = w.cascade_groups()
    gs_d, pre_d = torch.from_numpy(gs).cuda(), torch.from_numpy(pre).cuda()
    S = w.num_seqs
    mx, mp = int(w.context_lens.max()), int(pre.max())
    out = torch.empty_like(t["q"])
    ws = torch.empty(pkv.cascade_workspace_size(S, 32, 128, mx, mp), dtype=torch.uint8,
                     device="cuda")

    def step():
        pkv.paged_attention_decode_cascade(out, t["q"], t["kc"], t["vc"], t["bt"], t["cl"],
                                           gs_d, pre_d, w.scale, max_context_len=mx,
                                           max_prefix_len=mp, workspace=ws,
                                           device_errors=t["err"])
    pkv.reshape_and_cache(t["k_new"], t["v_new"], t["kc"], t["vc"], t["slots"])
    replay_matches_eager(step, t, out)


def test_mixed_batch_in_a_graph():
    w = workloads.mixed(seed=9, num_decode=8, num_prefill=2, chunk=200, prior=300)
    t = setup(w)
    nd = 8
    out = torch.empty_like(t["q"])
    mx = int(w.context_lens.max())
    ws = torch.empty(max(256, pkv.mixed_workspace_size(nd, t["q"].shape[0], 32, 128, mx)),
                     dtype=torch.uint8, device="cuda")

    def step():
        pkv.reshape_and_cache(t["k_new"], t["v_new"], t["kc"], t["vc"], t["slots"],
                              device_errors=t["err"])
        pkv.paged_attention_mixed(out, t["q"], t["kc"], t["vc"], t["bt"], t["cl"], t["qsl"], nd,
                                  w.scale, max_q_len=200, max_context_len=mx, workspace=ws,
                                  device_errors=t["err"])
    replay_matches_eager(step, t, out)
