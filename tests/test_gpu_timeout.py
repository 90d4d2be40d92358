"""Failure detection on the GPU without a GPU fault: a device-side wait that
runs out.

The test hook pkv_debug_arm_wait_timeout makes the next attention call's
first CTA skip one tile copy (it is never issued, so nothing is left in
flight) and bounds every device wait by a short limit.  The waits for that
tile give up, the kernel flags PKV_DEVERR_TIMEOUT, finishes or waits out its
own copies and MMAs, frees its tensor memory and returns; pkv_check_errors
reports PKV_ERR_TIMEOUT.  A normal call on the same device afterwards must
match the oracle again.  Nothing here traps, faults or hangs: every wait in
the kernels is bounded.
"""
import ctypes

import pytest
import torch

import paged_kv_cache_98_gb300 as pkv
import workloads
from _gpu import bits_to_dev, cache_tensors, decode_inputs, fill_device_cache, prefill_inputs
from test_gpu_parity import run_case

pytestmark = pytest.mark.gpu
F16, BF16 = workloads.F16, workloads.BF16
TIMEOUT_BIT = 0x8   # PKV_DEVERR_TIMEOUT
LIMIT_US = 20000    # 20 ms per wait instead of about 2 s


@pytest.fixture(scope="module", autouse=True)
def _library():
    from paged_kv_cache_98_gb300 import _build
    _build.build()
    pkv.load()


def _device_state(w):
    k, v, q = workloads.values_cpu(w)
    kc, vc = cache_tensors(w)
    fill_device_cache(w, bits_to_dev(k, w.src_dtype), bits_to_dev(v, w.src_dtype), kc, vc)
    return kc, vc, bits_to_dev(q, w.q_dtype)


def _decode_times_out(w, skip):
    kc, vc, qd = _device_state(w)
    ids, qq, bt, cl = decode_inputs(w, qd)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(qq)
    pkv.debug_arm_wait_timeout(skip, LIMIT_US)
    pkv.paged_attention_decode(out, qq, kc, vc, bt, cl, w.scale,
                               max_context_len=int(w.context_lens[ids].max()), device_errors=err)
    bits = ctypes.c_uint32(0)
    rc = pkv.load().pkv_check_errors(ctypes.c_void_p(err.data_ptr()), ctypes.byref(bits), None)
    assert rc == -6, pkv.status_string(rc)  # PKV_ERR_TIMEOUT
    assert bits.value & TIMEOUT_BIT
    # the hook was taken by that call: the same call again is clean
    pkv.paged_attention_decode(out, qq, kc, vc, bt, cl, w.scale,
                               max_context_len=int(w.context_lens[ids].max()), device_errors=err)
    assert pkv.check_errors(err) == 0


@pytest.mark.parametrize("skip", [1, 3])
def test_tensor_core_decode_wait_runs_out(skip):
    # g = 4, head_dim 128: the tcgen05 decode kernel; several partitions
    w = workloads.independent("timeout-tc", 7101, [1300, 40, 2000, 700], 16, 4, 128, BF16, BF16)
    _decode_times_out(w, skip)
    assert run_case(w) > 0  # the device is healthy and the kernel correct afterwards


def test_tensor_core_prefill_wait_runs_out():
    w = workloads.independent("timeout-pre", 7103, [900, 1500, 300], 16, 4, 128, BF16, BF16,
                              q_lens=[256, 300, 64])
    kc, vc, qd = _device_state(w)
    ids, qq, bt, cl, qsl = prefill_inputs(w, qd)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(qq)
    pkv.debug_arm_wait_timeout(2, LIMIT_US)
    pkv.paged_attention_prefill_chunk(out, qq, kc, vc, bt, cl, qsl, w.scale,
                                      max_q_len=int(w.q_lens[ids].max()),
                                      max_context_len=int(w.context_lens[ids].max()),
                                      device_errors=err)
    assert pkv.check_errors(err) & TIMEOUT_BIT
    assert run_case(w) > 0


def test_hook_rejects_nonpositive_index():
    with pytest.raises(pkv.PagedKVError):
        pkv.debug_arm_wait_timeout(0, LIMIT_US)
