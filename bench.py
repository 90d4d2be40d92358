#!/usr/bin/env python3
"""Paged KV-cache decode benchmark on one GB300: KV-read GB/s (fraction of the
measured HBM peak) and attended tokens/s.

A step is one pass of the hot path over one batch: the cache write of the
step's new K/V (reshape_and_cache through the slot mapping), then paged decode
attention of every sequence (split-K partitions plus the log-sum-exp merge).
The headline workload is the LLaMA-2-7B-shaped decode: 64 sequences x 4096
tokens, 32 q = 32 kv heads, head_dim 128, bf16, 16-token blocks scattered over
a pool of 1.25x the demand.  Its 4.3 GB of K/V per step exceed the 129 MB L2,
so consecutive steps read from HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica on its own GPU (the path has no cross-GPU exchange); the time is the
max over ranks and the value counts the bytes of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode KV-read GB/s (% of GB300 HBM peak) and attended tokens/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # NVIDIA's GB300 HBM3e figure, context only (not measured here)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--no-also", action="store_true", help="skip the other workloads")
    ap.add_argument("--mixed-entry", default="separate", choices=["separate", "fused"],
                    help="a batch with decode rows and chunks: separate decode and prefill "
                         "calls, or one pkv_paged_attention_mixed call")
    ap.add_argument("--decode-entry", default="plain", choices=["plain", "cascade"],
                    help="decode through pkv_paged_attention_decode or, reading each shared "
                         "prompt block once per group, pkv_paged_attention_decode_cascade")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only", choices=["tree_verify", "copy_blocks"],
                    help="run one of the side measurements alone and print its JSON (profiling)")
    ap.add_argument("--workload", default="llama2_7b",
                    help="named workload of the timed step (default: the LLaMA-2-7B-shaped "
                         "decode); the others are for profiling one workload alone")
    return ap.parse_args()


# ---- environment -----------------------------------------------------------------
# ncu summaries under profiles/ whose recorded DRAM traffic belongs to the decode
# kernel of each workload (other workloads report no traffic)
TRAFFIC_PROFILES = {
    "llama2_7b": "decode_llama2_7b",
    "gqa70b_shared": "decode_gqa70b_shared_tc",
    "long_fp8": "decode_long_fp8_tc",
    "gqa70b_shared+cascade": "decode_gqa70b_shared_cascade",
}


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The largest of the ranks' values, on every rank (x itself without a
    process group): step times are taken as the slowest replica's."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_hash(files) -> str:
    """sha256 (16 hex digits) of the named files under paged_kv_cache_98_gb300/csrc."""
    h = hashlib.sha256()
    for name in sorted(files):
        with open(os.path.join(ROOT, "paged_kv_cache_98_gb300", "csrc", name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(name: str):
    """DRAM bytes per full launch from an ncu capture summarised in
    profiles/<name>.md (lines 'traffic_bytes_per_launch: X', 'src_files: a b ...',
    'src_sha: H'); None when absent or when those kernel sources have changed."""
    path = os.path.join(ROOT, "profiles", name + ".md")
    try:
        text = open(path, encoding="utf-8").read()
    except OSError:
        return None
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    f = re.search(r"src_files:\s*(.+)", text)
    h = re.search(r"src_sha:\s*([0-9a-f]+)", text)
    if not (t and f and h):
        return None
    try:
        if source_hash(f.group(1).split()) != h.group(1):
            return None
    except OSError:
        return None
    return float(t.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- one workload on the GPU ---------------------------------------------------------
class GpuStep:
    """Device-resident state of one workload and its step (cache write, decode
    attention, and prefill-chunk attention when the workload has chunks)."""

    def __init__(self, w, dev, cascade=False, fused=False):
        import numpy as np
        import torch

        import paged_kv_cache_98_gb300 as pkv
        import workloads

        self.w, self.dev, self.pkv = w, dev, pkv
        k, v, q = workloads.values_device(w, dev)
        self.ks = self.vs = 1.0
        if w.kv_dtype == workloads.E4M3:
            # per-tensor scales amax / 448 of the source tensors
            self.ks = float(np.float32(k.float().abs().max().item()) / np.float32(448.0))
            self.vs = float(np.float32(v.float().abs().max().item()) / np.float32(448.0))
        shape = (w.num_blocks, w.num_kv_heads, 16, w.head_dim)
        cdt = torch.uint8 if w.kv_dtype == workloads.E4M3 else k.dtype
        self.kc = torch.zeros(shape, dtype=cdt, device=dev)
        self.vc = torch.zeros(shape, dtype=cdt, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        chunk = 1 << 16
        for a in range(0, len(w.fill_rows), chunk):
            r = torch.from_numpy(w.fill_rows[a:a + chunk]).to(dev)
            pkv.reshape_and_cache(k.index_select(0, r).contiguous(), v.index_select(0, r).contiguous(),
                                  self.kc, self.vc, torch.from_numpy(w.fill_slots[a:a + chunk]).to(dev),
                                  self.ks, self.vs, device_errors=self.err)
        r = torch.from_numpy(w.new_rows).to(dev)
        self.k_new = k.index_select(0, r).contiguous()
        self.v_new = v.index_select(0, r).contiguous()
        self.slots = torch.from_numpy(w.new_slots).to(dev)
        qsl = workloads.query_start_loc(w.q_lens)
        self.dec = w.decode_ids()
        self.pre = w.prefill_ids()
        self.q_dec = q.index_select(0, torch.from_numpy(qsl[self.dec].astype(np.int64)).to(dev)).contiguous()
        self.bt = torch.from_numpy(np.ascontiguousarray(w.block_tables[self.dec])).to(dev)
        self.cl = torch.from_numpy(np.ascontiguousarray(w.context_lens[self.dec])).to(dev)
        self.max_ctx = int(w.context_lens[self.dec].max()) if len(self.dec) else 0
        self.out = torch.empty_like(self.q_dec)
        S, H, D = self.q_dec.shape
        self.ws_bytes = pkv.decode_workspace_size(S, H, D, self.max_ctx, 0)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.parts = max(1, -(-self.max_ctx // 512))
        if len(self.pre):
            rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in self.pre]).astype(np.int64)
            self.q_pre = q.index_select(0, torch.from_numpy(rows).to(dev)).contiguous()
            self.bt_pre = torch.from_numpy(np.ascontiguousarray(w.block_tables[self.pre])).to(dev)
            self.cl_pre = torch.from_numpy(np.ascontiguousarray(w.context_lens[self.pre])).to(dev)
            self.qsl_pre = torch.from_numpy(workloads.query_start_loc(w.q_lens[self.pre])).to(dev)
            self.max_q_pre = int(w.q_lens[self.pre].max())
            self.max_ctx_pre = int(w.context_lens[self.pre].max())
            self.out_pre = torch.empty_like(self.q_pre)
            nb = pkv.prefill_workspace_size(self.q_pre.shape[0], H, D, self.max_ctx_pre,
                                            self.max_q_pre)
            self.ws_pre = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
        self.has_mixed = len(self.dec) > 0 and len(self.pre) > 0
        self.fused = fused and self.has_mixed
        if self.has_mixed:
            # one call over the whole batch (the workload lists its decode rows first)
            nd = len(self.dec)
            assert np.array_equal(self.dec, np.arange(nd))
            self.q_all = q.contiguous()
            self.bt_all = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(dev)
            self.cl_all = torch.from_numpy(np.ascontiguousarray(w.context_lens)).to(dev)
            self.qsl_all = torch.from_numpy(qsl).to(dev)
            self.out_all = torch.empty_like(self.q_all)
            self.max_ctx_all = int(w.context_lens.max())
            nb = pkv.mixed_workspace_size(nd, self.q_all.shape[0], H, D, self.max_ctx_all)
            self.ws_all = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
        self.cascade = cascade
        if cascade:
            gs, pre = w.cascade_groups()
            self.casc_mp = int(pre.max()) if len(pre) else 0
            self.casc_ws = torch.empty(
                max(256, pkv.cascade_workspace_size(S, H, D, self.max_ctx, self.casc_mp)),
                dtype=torch.uint8, device=dev)
            self.casc_gs = torch.from_numpy(gs).to(dev)
            self.casc_pre = torch.from_numpy(pre).to(dev)
        del k, v, q
        torch.cuda.synchronize(dev)
        if pkv.check_errors(self.err) != 0:
            raise RuntimeError("device-side checks failed while filling the cache")

    def cascade_timed(self, steps: int, warmup: int) -> float:
        """Mean CUDA-event time (ms) of the decode through the cascade entry
        point; its output is checked against the plain decode's."""
        import torch
        gs, pre = self.w.cascade_groups()
        gs_d = torch.from_numpy(gs).to(self.dev)
        pre_d = torch.from_numpy(pre).to(self.dev)
        S, H, D = self.q_dec.shape
        mp = int(pre.max()) if len(pre) else 0
        ws = torch.empty(max(256, self.pkv.cascade_workspace_size(S, H, D, self.max_ctx, mp)),
                         dtype=torch.uint8, device=self.dev)
        out = torch.empty_like(self.out)

        def one():
            self.pkv.paged_attention_decode_cascade(
                out, self.q_dec, self.kc, self.vc, self.bt, self.cl, gs_d, pre_d, self.w.scale,
                max_context_len=self.max_ctx, max_prefix_len=mp, workspace=ws,
                device_errors=self.err)
        for _ in range(warmup):
            one()
        self.decode()
        torch.cuda.synchronize(self.dev)
        if (out.float() - self.out.float()).abs().max().item() > 0.05:
            raise RuntimeError("cascade decode disagrees with plain decode")
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(steps):
            one()
        t1.record()
        torch.cuda.synchronize(self.dev)
        return t0.elapsed_time(t1) / steps

    def launches_per_step(self) -> int:
        n = 1  # cache write
        if self.fused:
            return n + 1 + (1 if self.parts > 1 else 0)  # fused attention, decode merge
        if len(self.dec) and self.cascade:
            n += 3  # shared-prefix pass, own-keys decode, merge
        elif len(self.dec):
            n += 1 + (1 if self.parts > 1 else 0)
        if len(self.pre):
            # the tensor-core chunk kernel (after the query split on E4M3 caches)
            n += 1 + (1 if self.w.kv_dtype == 2 else 0)
        return n

    def write(self):
        self.pkv.reshape_and_cache(self.k_new, self.v_new, self.kc, self.vc, self.slots, self.ks,
                                   self.vs, device_errors=self.err)

    def mixed(self):
        self.pkv.paged_attention_mixed(
            self.out_all, self.q_all, self.kc, self.vc, self.bt_all, self.cl_all, self.qsl_all,
            len(self.dec), self.w.scale, max_q_len=self.max_q_pre,
            max_context_len=self.max_ctx_all, workspace=self.ws_all, device_errors=self.err)

    def fused_timed(self, steps: int, warmup: int) -> float:
        """Mean CUDA-event time (ms) of the whole batch's attention in one
        pkv_paged_attention_mixed call; its output is checked against the
        separate decode and prefill calls' (they run the same arithmetic)."""
        import torch
        fused, self.fused = self.fused, False
        for _ in range(warmup):
            self.mixed()
        self.decode()
        self.prefill()
        self.fused = fused
        torch.cuda.synchronize(self.dev)
        nd = len(self.dec)
        if not (torch.equal(self.out_all[:nd], self.out) and
                torch.equal(self.out_all[nd:], self.out_pre)):
            raise RuntimeError("fused mixed-batch attention disagrees with the separate calls")
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(steps):
            self.mixed()
        t1.record()
        torch.cuda.synchronize(self.dev)
        return t0.elapsed_time(t1) / steps

    def decode(self):
        if self.fused:
            self.mixed()
            return
        if len(self.dec) and self.cascade:
            self.pkv.paged_attention_decode_cascade(
                self.out, self.q_dec, self.kc, self.vc, self.bt, self.cl, self.casc_gs,
                self.casc_pre, self.w.scale, max_context_len=self.max_ctx,
                max_prefix_len=self.casc_mp, workspace=self.casc_ws, device_errors=self.err)
        elif len(self.dec):
            self.pkv.paged_attention_decode(
                self.out, self.q_dec, self.kc, self.vc, self.bt, self.cl, self.w.scale,
                max_context_len=self.max_ctx, k_scale=self.ks, v_scale=self.vs, workspace=self.ws,
                device_errors=self.err)

    def prefill(self):
        if len(self.pre) and not self.fused:
            self.pkv.paged_attention_prefill_chunk(
                self.out_pre, self.q_pre, self.kc, self.vc, self.bt_pre, self.cl_pre, self.qsl_pre,
                self.w.scale, max_q_len=self.max_q_pre, max_context_len=self.max_ctx_pre,
                k_scale=self.ks, v_scale=self.vs, workspace=self.ws_pre, device_errors=self.err)

    def step(self):
        self.write()
        self.decode()
        self.prefill()

    def timed(self, steps: int, warmup: int, barrier=None):
        """Times exactly `steps` steps with one event pair around them (the
        contract's timed region), then a second pass with events around each
        call for the per-kernel breakdown."""
        import torch
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize(self.dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        if barrier:
            barrier()
        torch.cuda.synchronize(self.dev)
        t0.record()
        for _ in range(steps):
            self.step()
        t1.record()
        torch.cuda.synchronize(self.dev)
        if barrier:
            barrier()
        total = t0.elapsed_time(t1)
        n = max(1, min(steps, 200))
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
        for e in ev:
            e[0].record()
            self.write()
            e[1].record()
            self.decode()
            e[2].record()
            self.prefill()
            e[3].record()
        torch.cuda.synchronize(self.dev)
        dec = [e[1].elapsed_time(e[2]) for e in ev]
        pre = [e[2].elapsed_time(e[3]) for e in ev]
        wr = [e[0].elapsed_time(e[1]) for e in ev]
        return {"total_ms": total, "decode_ms": statistics.mean(dec),
                "prefill_ms": statistics.mean(pre), "write_ms": statistics.mean(wr),
                "decode_ms_median": statistics.median(dec)}

    def e2e(self, steps: int, warmup: int):
        """Same step through the public API from pinned host buffers: every step
        copies its inputs in and reads its outputs back, inside the timed
        region.  The copies are pipelined as a server would run them: inputs
        go to one of two device buffer sets on a copy stream while the
        previous step computes, and outputs come back on a third stream."""
        import torch
        names = ["k_new", "v_new", "slots", "q_dec", "bt", "cl"]
        if len(self.pre):
            names += ["q_pre", "bt_pre", "cl_pre", "qsl_pre"]
        if self.fused:
            names = ["k_new", "v_new", "slots", "q_all", "bt_all", "cl_all", "qsl_all"]
        if self.cascade:
            names += ["casc_gs", "casc_pre"]
        outs = ["out_all"] if self.fused else ["out"] + (["out_pre"] if len(self.pre) else [])
        sets = [{n: getattr(self, n) for n in names + outs},
                {n: torch.empty_like(getattr(self, n)) for n in names + outs}]
        host_in = {}
        for n in names:
            h = torch.empty(getattr(self, n).shape, dtype=getattr(self, n).dtype, pin_memory=True)
            h.copy_(getattr(self, n))
            host_in[n] = h
        host_out = [{n: torch.empty(sets[0][n].shape, dtype=sets[0][n].dtype, pin_memory=True)
                     for n in outs} for _ in range(2)]
        h2d = sum(h.numel() * h.element_size() for h in host_in.values())
        d2h = sum(h.numel() * h.element_size() for h in host_out[0].values())
        comp = torch.cuda.current_stream(self.dev)
        s_in, s_out = torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev)
        ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "comp", "out")}
        used = [False, False]

        def run(i):
            b = i & 1
            with torch.cuda.stream(s_in):
                if used[b]:
                    s_in.wait_event(ev["comp"][b])  # step i - 2 has read set b's inputs
                for n in names:
                    sets[b][n].copy_(host_in[n], non_blocking=True)
                ev["in"][b].record(s_in)
            comp.wait_event(ev["in"][b])
            if used[b]:
                comp.wait_event(ev["out"][b])  # set b's outputs have been read back
            for n, t in sets[b].items():
                setattr(self, n, t)
            self.step()
            ev["comp"][b].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["comp"][b])
                for n in outs:
                    host_out[b][n].copy_(sets[b][n], non_blocking=True)
                ev["out"][b].record(s_out)
            used[b] = True

        def drain():
            for b in range(2):
                if used[b]:
                    comp.wait_event(ev["out"][b])

        for i in range(warmup):
            run(i)
        drain()
        torch.cuda.synchronize(self.dev)
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        a.record(comp)
        s_in.wait_stream(comp)
        s_out.wait_stream(comp)
        for i in range(steps):
            run(warmup + i)
        drain()
        z.record(comp)
        torch.cuda.synchronize(self.dev)
        last = host_out[(warmup + steps - 1) & 1]
        for n, t in sets[0].items():
            setattr(self, n, t)
        # the pipelined results are the step's results
        self.step()
        torch.cuda.synchronize(self.dev)
        for n in outs:
            if not torch.equal(last[n].view(torch.uint8), getattr(self, n).cpu().view(torch.uint8)):
                raise RuntimeError("pipelined end-to-end step returned a different " + n)
        return a.elapsed_time(z) / steps, h2d, d2h


def unique_kv_bytes(w) -> int:
    import numpy as np
    blocks = set()
    for s in w.decode_ids():
        nb = -(-int(w.context_lens[s]) // 16)
        blocks.update(w.block_tables[s, :nb].tolist())
    return len(blocks) * 16 * 2 * w.num_kv_heads * w.head_dim * w.kv_elem_bytes


def describe(w) -> str:
    import numpy as np
    dt = {0: "fp16", 1: "bf16", 2: "fp8-e4m3"}
    ctx = w.context_lens[w.decode_ids()]
    return (f"{w.name}: {len(ctx)} decode seqs (ctx {int(ctx.min())}..{int(ctx.max())}, "
            f"mean {float(np.mean(ctx)):.0f}), {w.num_heads} q / {w.num_kv_heads} kv heads, "
            f"head_dim {w.head_dim}, block 16, q {dt[w.q_dtype]}, kv {dt[w.kv_dtype]}"
            + (f", {len(w.prefill_ids())} prefill chunks of {int(w.q_lens[w.prefill_ids()].max())}"
               if len(w.prefill_ids()) else ""))


# ---- CPU oracle ------------------------------------------------------------------------
class OracleSample:
    """The oracle's cache write + decode on a sample shaped like the workload
    (context ctx, H/Hkv heads, head_dim D): `nseq` sequences, `groups` KV heads
    each.  Set-up (drawing values, filling the host cache) is not timed."""

    def __init__(self, H, Hkv, D, ctx, kv_dtype, nseq, groups):
        import numpy as np

        import oracle
        import workloads
        self.o, self.np = oracle, np
        g = H // Hkv
        self.kv_dtype = kv_dtype
        w = workloads.independent("cpu sample", 77, [ctx] * nseq, g * groups, groups, D,
                                  workloads.BF16, kv_dtype)
        self.w = w
        k, v, q = workloads.values_cpu(w)
        eb = 1 if kv_dtype == workloads.E4M3 else 2
        self.kc = np.zeros(w.num_blocks * groups * 16 * D * eb, np.uint8)
        self.vc = np.zeros_like(self.kc)
        self.sc = 0.01 if kv_dtype == workloads.E4M3 else 1.0
        oracle.reshape_and_cache(np.ascontiguousarray(k[w.fill_rows]),
                                 np.ascontiguousarray(v[w.fill_rows]), self.kc, self.vc,
                                 w.fill_slots, w.num_blocks, 16, workloads.BF16, kv_dtype,
                                 self.sc, self.sc)
        self.k_new = np.ascontiguousarray(k[w.new_rows])
        self.v_new = np.ascontiguousarray(v[w.new_rows])
        self.q = np.ascontiguousarray(q)
        self.bytes = w.kv_read_bytes()
        self.desc = (f"{nseq} sequence(s) x {ctx} tokens, {groups} of {Hkv} kv heads "
                     f"(x{g} q heads), head_dim {D}")

    def step(self) -> float:
        w, o = self.w, self.o
        t0 = time.perf_counter()
        o.reshape_and_cache(self.k_new, self.v_new, self.kc, self.vc, w.new_slots, w.num_blocks,
                            16, 1, self.kv_dtype, self.sc, self.sc)
        o.paged_attention_decode(self.q, self.kc, self.vc, w.block_tables, w.context_lens,
                                 w.num_kv_heads, w.head_dim, 16, w.num_blocks, w.scale, 1,
                                 self.kv_dtype, self.sc, self.sc)
        return time.perf_counter() - t0


def parallel_oracle_seconds(smp: "OracleSample", threads: int, reps: int = 3) -> float:
    """The same oracle decode over the sample's sequences split across host
    threads (the oracle's C calls release the interpreter lock), best of reps."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np
    w, o = smp.w, smp.o
    parts = [p for p in np.array_split(np.arange(w.num_seqs), threads) if len(p)]
    qsl = np.arange(w.num_seqs)

    def run(ids):
        o.paged_attention_decode(np.ascontiguousarray(smp.q[qsl[ids]]), smp.kc, smp.vc,
                                 w.block_tables[ids], w.context_lens[ids], w.num_kv_heads,
                                 w.head_dim, 16, w.num_blocks, w.scale, 1, smp.kv_dtype, smp.sc,
                                 smp.sc)

    best = float("inf")
    with ThreadPoolExecutor(len(parts)) as ex:
        for _ in range(reps):
            t0 = time.perf_counter()
            list(ex.map(run, parts))
            best = min(best, time.perf_counter() - t0)
    return best


def host_cpu() -> dict:
    """Host core count and CPU model, for the CPU baselines."""
    import platform
    model = platform.processor() or platform.machine()
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
                if line.lower().startswith("cpu part"):  # Arm: the part number
                    part = line.split(":", 1)[1].strip()
                    model = {"0xd4f": "Arm Neoverse V2"}.get(part, "Arm") + f" (part {part})"
                    break
    except OSError:
        pass
    return {"nproc": os.cpu_count(), "cpu": model, "arch": platform.machine()}


def oracle_sample(w, budget_s: float) -> OracleSample:
    """The largest sample (KV heads of one sequence, then whole sequences) whose
    step takes about budget_s on one core."""
    H, Hkv, D = w.num_heads, w.num_kv_heads, w.head_dim
    ctx = int(w.context_lens.max())
    probe = OracleSample(H, Hkv, D, ctx, w.kv_dtype, 1, 1)
    per_group = min(probe.step(), probe.step())
    groups = int(max(1, min(Hkv, budget_s / max(per_group, 1e-6))))
    nseq = 1
    if groups == Hkv:
        nseq = int(max(1, min(w.num_seqs, budget_s / max(per_group * Hkv, 1e-6))))
    return OracleSample(H, Hkv, D, ctx, w.kv_dtype, nseq, groups)


# ---- main ----------------------------------------------------------------------------------
def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    import workloads

    if args.impl == "reference":
        if rank != 0:
            return
        return reference_arm(args, world)

    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import paged_kv_cache_98_gb300 as pkv
    from paged_kv_cache_98_gb300 import _build
    if rank == 0 or world == 1:
        _build.build()
    if dist:
        dist.barrier()
    pkv.load()

    def barrier():
        if dist:
            dist.barrier()

    if args.only:
        peak, _ = hbm_peak()
        fn = tree_verify_rate if args.only == "tree_verify" else copy_blocks_rate
        print(json.dumps({"only": args.only, **fn(dev, peak)}), flush=True)
        return
    w = workloads.NAMED[args.workload]()
    cascade = args.decode_entry == "cascade"
    st = GpuStep(w, dev, cascade=cascade, fused=args.mixed_entry == "fused")
    sampler = ClockSampler(local).start()
    time.sleep(0.3)
    res = st.timed(args.steps, args.warmup, barrier)
    clocks = sampler.stop()
    total = max_over_ranks(res["total_ms"], dist, dev)
    if pkv.check_errors(st.err) != 0:
        raise RuntimeError("device-side checks failed during the timed steps")
    ms = total / args.steps
    kv_bytes = w.kv_read_bytes()
    tokens = int(w.context_lens.astype("int64").sum())
    value = world * kv_bytes / (ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    dec_ms = res["decode_ms"]
    # the cascade reads each shared prompt block once per group: its
    # algorithmic bytes are the unique K/V bytes
    alg_bytes = unique_kv_bytes(w) if cascade else kv_bytes
    achieved = alg_bytes / (dec_ms * 1e-3) / 1e9
    e2e_ms, h2d, d2h = st.e2e(max(20, min(args.steps, 200)), 5)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {0: "f16", 1: "bf16"}[w.q_dtype] + ("+e4m3-kv" if w.kv_dtype == 2 else ""),
        "data": "synthetic: seeded N(0,1) bf16 K/V/Q, block tables a seeded random permutation "
                "of a pool 1.25x the demand",
        "config": {
            "workload": describe(w),
            "num_seqs": w.num_seqs, "context": int(w.context_lens.max()),
            "num_heads": w.num_heads, "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": 16, "partition": 512, "pool_blocks": w.num_blocks,
            "decode_entry": args.decode_entry, "mixed_entry": args.mixed_entry,
            "kv_bytes_per_step": kv_bytes,
            "l2": f"inputs larger than L2: {kv_bytes / 1e9:.2f} GB of K/V read per step "
                  "vs 129 MB L2",
            "parallelism": f"replicas x{world}",
        },
        "attended_tokens_per_s": round(world * tokens / (ms * 1e-3), 1),
        "sequences_per_s": round(world * w.num_seqs / (ms * 1e-3), 1),
        "hbm_frac": round(world * alg_bytes / (ms * 1e-3) / 1e9 / world / peak, 4),
        "roofline": {
            "kernel": ("cascade decode (shared-prefix pass + own-keys decode + merge launches)"
                       if cascade else
                       "paged decode attention (attention + log-sum-exp merge launches)"),
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
            "peak_kind": f"{peak_kind} HBM copy bandwidth",
            "unit": "GB/s", "frac": round(achieved / peak, 4),
            "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
            "traffic": recorded_traffic(TRAFFIC_PROFILES.get(
                args.workload + ("+cascade" if cascade else ""), "")),
            "algorithmic_bytes_per_launch": alg_bytes,
            "decode_ms": round(dec_ms, 5), "write_ms": round(res["write_ms"], 5),
        },
        "e2e": {"value": round(world * kv_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": st.launches_per_step() * args.steps,
        "clocks": clocks,
    }
    del st
    torch.cuda.empty_cache()
    if not args.no_also and args.workload == "llama2_7b":
        line["also"] = other_workloads(dev, peak, barrier)
        line["also"]["tree_verify"] = tree_verify_rate(dev, peak)
        line["also"]["copy_blocks"] = copy_blocks_rate(dev, peak)
        line["also"]["host_block_pool"] = host_pool_rate()
    if rank == 0 and not args.no_cpu:
        smp = oracle_sample(w, args.cpu_seconds)
        secs = smp.step()
        line["cpu_baseline"] = {"value": round(smp.bytes / secs / 1e9, 4), "unit": "GB/s",
                                "cores": 1, "kind": "oracle", "sample": smp.desc,
                                "seconds": round(secs, 2), "host": host_cpu()}
        # the same oracle functions over the sample's sequences on every host core
        threads = max(1, min(os.cpu_count() or 1, smp.w.num_seqs))
        psecs = parallel_oracle_seconds(smp, threads)
        line["cpu_baseline_parallel"] = {
            "value": round(smp.bytes / psecs / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle, sequences split over threads", "sample": smp.desc,
            "seconds": round(psecs, 3)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def tree_verify_rate(dev, peak, reps: int = 50) -> dict:
    """Draft-tree verification at serving size: 128 sequences with the 70B-GQA head
    shape (64 q / 8 kv heads), contexts lognormal around 2000 tokens, each with a
    random 64-token draft tree, in one pkv_paged_attention_prefill_tree call."""
    import numpy as np
    import torch

    import paged_kv_cache_98_gb300 as pkv
    import workloads
    r = np.random.default_rng(77)
    prior = np.clip(np.exp(r.normal(np.log(2000.0), 1.0, size=128)).astype(int), 16, 12000)
    w = workloads.independent("tree-verify", 78, list(prior + 64), 64, 8, 128, workloads.BF16,
                              workloads.BF16, q_lens=[64] * 128)
    masks = np.concatenate([workloads.tree_mask(workloads.random_tree(r, 64))
                            for _ in range(128)])
    k, v, q = workloads.values_device(w, dev)
    kc = torch.zeros((w.num_blocks, 8, 16, 128), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    rows = torch.from_numpy(np.concatenate([w.fill_rows, w.new_rows])).to(dev)
    slots = torch.from_numpy(np.concatenate([w.fill_slots, w.new_slots])).to(dev)
    pkv.reshape_and_cache(k.index_select(0, rows).contiguous(),
                          v.index_select(0, rows).contiguous(), kc, vc, slots)
    bt = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(dev)
    cl = torch.from_numpy(np.ascontiguousarray(w.context_lens)).to(dev)
    qsl = torch.from_numpy(workloads.query_start_loc(w.q_lens)).to(dev)
    tm = torch.from_numpy(masks.view(np.int64)).to(dev)
    out = torch.empty_like(q)
    mx = int(w.context_lens.max())

    def call():
        pkv.paged_attention_prefill_tree(out, q, kc, vc, bt, cl, qsl, tm, w.scale, max_q_len=64,
                                         max_context_len=mx)
    for _ in range(3):
        call()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        call()
    z.record()
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(z) / reps
    kvb = w.kv_read_bytes(np.arange(w.num_seqs))  # every context token once per KV head
    # visible keys: the prior context for every draft token plus its ancestors in the tree
    vis = sum(int(w.context_lens[s] - 64) * 64 for s in range(128)) + \
        sum(bin(int(m)).count("1") for m in masks)
    flops = 4 * 64 * 128 * vis
    return {"workload": "128 draft trees of 64 tokens, 64 q / 8 kv heads, bf16, contexts "
                        f"{int(prior.min())}..{int(prior.max())} + 64",
            "ms": round(ms, 5), "kv_GBps": round(kvb / (ms * 1e-3) / 1e9, 1),
            "kv_frac": round(kvb / (ms * 1e-3) / 1e9 / peak, 4),
            "tflops": round(flops / (ms * 1e-3) / 1e12, 1), "kv_bytes": kvb}


def copy_blocks_rate(dev, peak, pairs: int = 4096, reps: int = 20) -> dict:
    """pkv_copy_blocks on a 70B-shaped pool (8 KV heads, head_dim 128, bf16: 32 KB
    per block and cache): `pairs` random disjoint (source, destination) pairs."""
    import numpy as np
    import torch

    import paged_kv_cache_98_gb300 as pkv
    nb = 4 * pairs
    kc = torch.zeros((nb, 8, 16, 128), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    perm = np.random.default_rng(11).permutation(nb).astype(np.int32)
    pr = torch.from_numpy(np.stack([perm[:pairs], perm[pairs:2 * pairs]], 1).copy()).to(dev)
    for _ in range(3):
        pkv.copy_blocks(kc, vc, pr)
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        pkv.copy_blocks(kc, vc, pr)
    z.record()
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(z) / reps
    moved = 2 * 2 * pairs * 8 * 16 * 128 * 2  # read + write, K and V
    return {"pairs": pairs, "ms": round(ms, 5), "GBps": round(moved / (ms * 1e-3) / 1e9, 1),
            "frac": round(moved / (ms * 1e-3) / 1e9 / peak, 4),
            "bytes_read_written": moved}


def host_pool_rate(requests: int = 20000) -> dict:
    """The host block pool: requests drawn from 16 shared prompts (200-2000
    tokens) arrive (prefix match + append of the rest), decode 16 tokens one at
    a time, and leave; requests per second on one host core."""
    import numpy as np

    import paged_kv_cache_98_gb300 as pkv
    r = np.random.default_rng(12)
    prompts = [r.integers(0, 32000, int(r.integers(200, 2001))).astype(np.int32)
               for _ in range(16)]
    pool = pkv.BlockPool(200000)
    live, hits, toks = [], 0, 0
    t0 = time.perf_counter()
    for i in range(requests):
        p = np.concatenate([prompts[i % 16], r.integers(0, 32000, 20).astype(np.int32)])
        req = pool.request()
        m = req.match_prefix(p)
        hits += m
        req.append(p[m:])
        toks += len(p)
        for j in range(16):
            req.append(p[j:j + 1])
        live.append(req)
        if len(live) > 64:
            live.pop(0).free()
    sec = time.perf_counter() - t0
    for q in live:
        q.free()
    pool.close()
    return {"requests": requests, "seconds": round(sec, 3),
            "requests_per_s": round(requests / sec, 1),
            "prefix_hit_frac": round(hits / toks, 4), "cores": 1,
            "note": "through the Python binding: 18 library calls per request"}


def other_workloads(dev, peak, barrier):
    """The other named workloads, each timed the same way (fewer steps)."""
    import torch

    import workloads
    out = {}
    for name, steps in (("gqa70b_shared", 200), ("long_fp8", 100), ("mixed", 100),
                        ("mixed_fp8", 100)):
        w = workloads.NAMED[name]()
        st = GpuStep(w, dev)
        res = st.timed(steps, 5, barrier)
        ms = res["total_ms"] / steps
        kvb = w.kv_read_bytes()
        d = {"workload": describe(w), "ms_per_step": round(ms, 5),
             "decode_ms": round(res["decode_ms"], 5),
             "decode_GBps_logical": round(kvb / (res["decode_ms"] * 1e-3) / 1e9, 1),
             "decode_frac_logical": round(kvb / (res["decode_ms"] * 1e-3) / 1e9 / peak, 4),
             "kv_bytes_logical": kvb,
             "attended_tokens_per_s": round(float(w.context_lens[w.decode_ids()].sum()) /
                                            (res["decode_ms"] * 1e-3), 1)}
        if name == "gqa70b_shared":
            ub = unique_kv_bytes(w)
            d["kv_bytes_unique"] = ub
            d["decode_GBps_unique"] = round(ub / (res["decode_ms"] * 1e-3) / 1e9, 1)
            # DRAM bytes of one decode launch from the recorded ncu capture (L2 serves
            # the repeated reads of shared blocks), while the kernel sources match it
            tr = recorded_traffic(TRAFFIC_PROFILES[name])
            if tr:
                d["decode_GBps_dram"] = round(tr / (res["decode_ms"] * 1e-3) / 1e9, 1)
                d["decode_frac_dram"] = round(tr / (res["decode_ms"] * 1e-3) / 1e9 / peak, 4)
            # the same decode through the cascade entry point (each shared prompt
            # block read once per group of samples)
            cms = st.cascade_timed(steps, 5)
            d["cascade_decode_ms"] = round(cms, 5)
            d["cascade_GBps_logical"] = round(kvb / (cms * 1e-3) / 1e9, 1)
            d["cascade_GBps_unique"] = round(ub / (cms * 1e-3) / 1e9, 1)
            d["cascade_speedup"] = round(res["decode_ms"] / cms, 3)
        if name == "mixed":  # (E4M3 caches have no fused kernel)
            # the same batch's attention in one fused call
            fms = st.fused_timed(steps, 5)
            d["fused_attention_ms"] = round(fms, 5)
            d["separate_attention_ms"] = round(res["decode_ms"] + res["prefill_ms"], 5)
            d["fused_speedup"] = round((res["decode_ms"] + res["prefill_ms"]) / fms, 3)
        if len(w.prefill_ids()):
            flops = 0
            for s in w.prefill_ids():
                c, ql = int(w.context_lens[s]), int(w.q_lens[s])
                keys = sum(c - ql + i + 1 for i in range(ql))
                flops += 4 * w.num_heads * w.head_dim * keys
            d["prefill_ms"] = round(res["prefill_ms"], 5)
            d["prefill_query_tokens_per_s"] = round(
                float(w.q_lens[w.prefill_ids()].sum()) / (res["prefill_ms"] * 1e-3), 1)
            d["prefill_tflops"] = round(flops / (res["prefill_ms"] * 1e-3) / 1e12, 2)
            d["prefill_flops"] = flops
        if pkv_errors(st):
            d["device_errors"] = True
        out[name] = d
        del st
        torch.cuda.empty_cache()
    return out


def pkv_errors(st) -> bool:
    return st.pkv.check_errors(st.err) != 0


def reference_arm(args, world):
    """The oracle, as it stands, on one host core: each step a bounded sample of
    the headline workload, sized so that the whole run takes a few minutes."""
    import workloads
    w = workloads.llama2_7b()
    steps, warm = args.steps, args.warmup
    budget = max(0.02, min(2.0, 150.0 / max(1, steps + warm)))
    smp = oracle_sample(w, budget)
    t0 = time.perf_counter()
    times = []
    for i in range(steps + warm):
        dt = smp.step()
        if i >= warm:
            times.append(dt)
    wall = time.perf_counter() - t0
    sec = statistics.mean(times) if times else smp.step()
    value = smp.bytes / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": steps, "warmup": warm, "ms_per_step": round(sec * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded N(0,1) bf16 K/V/Q (CPU draw), scattered block tables",
        "config": {"workload": describe(w), "sample_per_step": smp.desc},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": smp.desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s": round(wall, 1),
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
