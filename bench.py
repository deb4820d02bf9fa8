"""Benchmark of one speculative tree-verify round over a paged 3-bit KV cache.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long262k]
                    [--path exact|int8] [--impl ours|reference]

A step is one whole verify round of the workload: for each of the 16
attention layers, append the tree's T rows to the 3-bit cache
(stv_kv_append_pack), run the tree-masked split-KV verify attention
(stv_verify_attn) and merge its splits (stv_split_combine); then greedy tree
acceptance (stv_tree_accept) and compaction of the accepted rows in every
layer (stv_kv_commit).  The metric is microseconds per layer-round (the
round's time / 16), with the packed KV bytes the round streams per
layer-round and their rate (GB/s) against the HBM roofline.

Inputs are seeded synthetic tensors (workloads.py), resident in HBM before
the timed region.  The cache of 16 layers x 224 MiB (262K context) is far
larger than L2 (129 MB), so no flush is needed between steps.

Multi-GPU: the round does not need an exchange between GPUs, so N GPUs run N
independent replicas (one process per GPU under torchrun); value aggregates
their layer-rounds over the slowest rank's time.

--impl reference times the fp64 CPU oracle (the only other implementation of
this method that exists here) on the host cores, on a bounded sample of the
same workload, scaled to the same unit.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
METRIC = "verify-attn us/layer-round and HBM GB/s (% of roofline) at 32K and 262K ctx"
UNIT = "us/layer-round"


# Packed bytes per token and KV head, K + V: the 3-bit cache holds 96 B of
# codes and 16 B of fp16 group scales for each; the int4 per-token-head cache
# 128 B of codes and one 2 B scale; the K 4 / V 2-bit cache 128 B (K) and
# 64 B (V) of codes and 16 B of group scales each.
KV_FORMATS = {"bit3": (32, 2 * (96 + 16)), "int4": (256, 2 * (128 + 2)), "k4v2": (32, (128 + 16) + (64 + 16))}


def algorithmic_bytes_per_layer_round(ctx_list, t, hq=24, hkv=4, kv_format="bit3"):
    """Packed KV streamed by verify (every visible key's bytes over all KV
    heads) plus Q in and O out."""
    kv = sum(c + t for c in ctx_list) * hkv * KV_FORMATS[kv_format][1]
    qo = len(ctx_list) * 2 * t * hq * 256 * 2
    return kv + qo


def verify_kernel_bytes(ctx_list, t, hq=24, hkv=4, kv_format="bit3"):
    """Bytes one verify launch must read: packed KV of every visible key and Q."""
    return sum(c + t for c in ctx_list) * hkv * KV_FORMATS[kv_format][1] + len(ctx_list) * t * hq * 256 * 2


def verify_kernel_flops(ctx_list, t, hq=24):
    """Algorithmic FLOPs of one verify launch: Q.K^T and P.V over every
    visible key, 2 x 2 x hq x 256 per (node, key) (the tree mask's hidden
    keys counted, as the MMA tile computes them)."""
    return sum(c + t for c in ctx_list) * t * hq * 256 * 4


def launches_per_step(args, w: workloads.Workload) -> int:
    L = args.layers or w.layers
    per_layer = (1 if args.one_launch and args.path == "exact" else 2 if args.fuse_append else 3) + \
        (1 if args.path == "int8" else 0)
    return L * per_layer + 2


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBs", "hbm"):
                if k in d and d[k]:
                    v = d[k]
                    v = v.get("value", v.get("burst")) if isinstance(v, dict) else v
                    return float(v), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """SM clock, power and clock-event reasons sampled during the timed
    region, through NVML (read-only queries: nothing is changed on the GPU).
    A thread polls every 5 ms; the device is found by its PCI bus id, so the
    samples are the GPU this process runs on whatever CUDA_VISIBLE_DEVICES
    says.  Without NVML it falls back to `nvidia-smi -lms`."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.005):
        self.dev, self.period = device_index, period_s
        self.samples, self.max_mhz, self.source = [], None, None

    def _nvml_open(self):
        import ctypes

        import torch

        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit")
        pr = torch.cuda.get_device_properties(self.dev)
        bus = f"{getattr(pr, 'pci_domain_id', 0):08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0".encode()
        h = ctypes.c_void_p()
        if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByPciBusId")
        self.nv, self.h, self.ct = nv, h, ctypes
        self.reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or nv.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1 = SM clock
            self.max_mhz = float(mx.value)

    def _nvml_sample(self):
        ct, nv, h = self.ct, self.nv, self.h
        mhz, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        ok = nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz)) == 0
        nv.nvmlDeviceGetPowerUsage(h, ct.byref(mw))
        self.reasons_fn(h, ct.byref(rs))
        if ok:
            self.samples.append((float(mhz.value), mw.value / 1000.0, int(rs.value)))

    def __enter__(self):
        import threading

        self.stop = threading.Event()
        try:
            self._nvml_open()
            self._nvml_sample()  # one sample before the timed region starts
            self.source = "nvml"

            def run():
                while not self.stop.wait(self.period):
                    self._nvml_sample()

            self.thread = threading.Thread(target=run, daemon=True)
            self.thread.start()
        except Exception:
            self.thread = None
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.dev), "--query-gpu=clocks.sm,clocks.max.sm,power.draw",
                     "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE,
                    stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi"
            except Exception:
                self.proc = None
        return self

    def __exit__(self, *a):
        self.stop.set()
        if getattr(self, "thread", None) is not None:
            self.thread.join()
            self._nvml_sample()  # and one after it
            self.nv.nvmlShutdown()
        elif getattr(self, "proc", None) is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            for line in (out or "").strip().splitlines():
                f = [x.strip() for x in line.split(",")]
                try:
                    self.samples.append((float(f[0]), float(f[2]), 0))
                    self.max_mhz = float(f[1])
                except (ValueError, IndexError):
                    pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"], "samples": 0}
        reasons = sorted({n for _, _, r in self.samples for bit, n in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(m for m, _, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples),
                "power_w_max": max(w for _, w, _ in self.samples), "source": self.source}


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

class GpuRound:
    """All layers of one workload resident on the GPU, plus one round's inputs."""

    def __init__(self, w: workloads.Workload, p_accept: float, device, layers: int | None = None,
                 fuse_append: bool = False, group: int = 32, kv_format: int = 0, one_launch: bool = False):
        import torch

        import speculative_tree_verify_bit_gb300 as stv

        self.stv, self.torch, self.w, self.dev = stv, torch, w, device
        self.fuse_append = fuse_append
        self.one_launch = one_launch  # exact path: append, verify and merge in one launch per layer
        self.L = layers or w.layers
        self.T, self.hq, self.hkv = w.t_nodes, w.hq, w.hkv
        self.shape = stv.make_shape(self.hq, self.hkv, group, kv_format)
        self.pool_pages, tables = workloads.page_tables_for(w)
        self.tables = tables
        self.seqs = [stv.Seq(torch.as_tensor(t, device=device), c) for t, c in zip(tables, w.ctx)]
        self.ctx = list(w.ctx)
        rt = workloads.round_trees(w, p_accept)
        self.parent = torch.as_tensor(rt.parent, device=device)
        self.draft = torch.as_tensor(rt.draft, device=device)
        self.argmax = torch.as_tensor(rt.argmax, device=device)
        T, n = self.T, w.n_seqs
        self.layers, self.q, self.k_tree, self.v_tree = [], [], [], []
        row_seq_ctx = torch.cat([torch.full((c,), s, dtype=torch.int32, device=device) for s, c in enumerate(w.ctx)])
        row_pos_ctx = torch.cat([torch.arange(c, dtype=torch.int32, device=device) for c in w.ctx])
        self.row_seq = torch.cat([torch.full((T,), s, dtype=torch.int32, device=device) for s in range(n)])
        self.row_pos = torch.cat([torch.arange(c, c + T, dtype=torch.int32, device=device) for c in w.ctx])
        for l in range(self.L):
            seed = workloads.layer_seed(w, l)
            layer = stv.LayerCache.empty(self.pool_pages, self.hkv, device=device, group=group)
            ks, vs, kt, vt = [], [], [], []
            for s, c in enumerate(w.ctx):
                k, v = workloads.kv_rows(seed + 7919 * s, c + T, self.hkv, device=device)
                ks.append(k[:c]); vs.append(v[:c]); kt.append(k[c:]); vt.append(v[c:])
            kc, vc = torch.cat(ks).contiguous(), torch.cat(vs).contiguous()
            stv.stv_kv_append_pack(self.shape, layer, self.seqs, kc, vc, row_seq_ctx, row_pos_ctx)
            del kc, vc, ks, vs
            self.layers.append(layer)
            self.k_tree.append(torch.cat(kt).contiguous())
            self.v_tree.append(torch.cat(vt).contiguous())
            self.q.append(workloads.q_rows(seed, n, T, self.hq, device=device).contiguous())
        torch.cuda.synchronize()
        self.ws_bytes = stv.stv_verify_workspace_bytes(self.shape, self.seqs, T)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)  # zero counters (one-launch layers)
        self.o = torch.empty((n, T, self.hq, 256), dtype=torch.float16, device=device)
        self.n_commit = torch.zeros(n, dtype=torch.int32, device=device)
        self.path = torch.zeros((n, T), dtype=torch.int32, device=device)
        self.out_ids = torch.zeros((n, T), dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        # A round's inputs (Q, tree K/V rows, trees) and its results (commit
        # counts, accepted ids) each live in one device buffer, as a serving
        # engine stages them: one host-to-device copy per round in, one out.
        self.inputs, views = self._stage(self.q + self.k_tree + self.v_tree + [self.parent, self.draft, self.argmax])
        L = self.L
        self.q, self.k_tree, self.v_tree = views[:L], views[L:2 * L], views[2 * L:3 * L]
        self.parent, self.draft, self.argmax = views[3 * L:]
        self.outputs, (self.n_commit, self.out_ids) = self._stage([self.n_commit, self.out_ids])

    def _stage(self, tensors):
        """One contiguous device buffer holding copies of `tensors`, each
        256-byte aligned; returns it and the tensors' views into it."""
        torch = self.torch
        sizes = [t.numel() * t.element_size() for t in tensors]
        offs, at = [], 0
        for sz in sizes:
            offs.append(at)
            at += (sz + 255) // 256 * 256
        buf = torch.zeros(at, dtype=torch.uint8, device=self.dev)
        views = []
        for t, off, sz in zip(tensors, offs, sizes):
            v = buf[off:off + sz].view(t.dtype).view(t.shape)
            v.copy_(t)
            views.append(v)
        return buf, views

    def set_trees(self, p_accept: float):
        """Draw the round's trees for another acceptance probability into the
        same device buffers (a captured graph keeps reading them)."""
        import torch

        rt = workloads.round_trees(self.w, p_accept)
        self.parent.copy_(torch.as_tensor(rt.parent))
        self.draft.copy_(torch.as_tensor(rt.draft))
        self.argmax.copy_(torch.as_tensor(rt.argmax))
        torch.cuda.synchronize()

    def step(self, path, verify_events=None):
        stv = self.stv
        one = self.one_launch and path == "exact"
        for l in range(self.L):
            if one:  # append, verify and merge in one cooperative launch
                if verify_events is not None:
                    verify_events[l][0].record()
                stv.stv_append_verify_combine(self.shape, self.layers[l], self.seqs, self.k_tree[l], self.v_tree[l],
                                              self.q[l], self.parent, self.T, path, self.ws, self.o,
                                              dev_status=self.status)
                if verify_events is not None:
                    verify_events[l][1].record()
                continue
            if not self.fuse_append:
                stv.stv_kv_append_pack(self.shape, self.layers[l], self.seqs, self.k_tree[l], self.v_tree[l],
                                       self.row_seq, self.row_pos, dev_status=self.status)
            if verify_events is not None:
                verify_events[l][0].record()
            if self.fuse_append:  # the tree rows' append runs inside the verify launch
                stv.stv_append_verify_attn(self.shape, self.layers[l], self.seqs, self.k_tree[l], self.v_tree[l],
                                           self.q[l], self.parent, self.T, path, self.ws, dev_status=self.status)
            else:
                stv.stv_verify_attn(self.shape, self.layers[l], self.seqs, self.q[l], self.parent, self.T, path,
                                    self.ws, dev_status=self.status)
            if verify_events is not None:
                verify_events[l][1].record()
            stv.stv_split_combine(self.shape, self.seqs, self.T, self.ws, self.o)
        timed_tail = verify_events is not None and len(verify_events) > self.L
        if timed_tail:  # one more event pair: around acceptance and commit
            verify_events[self.L][0].record()
        stv.stv_tree_accept(self.parent, self.draft, self.argmax, self.n_commit, self.path, self.out_ids,
                            dev_status=self.status)
        stv.stv_kv_commit(self.shape, self.layers, self.seqs, self.T, self.n_commit, self.path,
                          dev_status=self.status)
        if timed_tail:
            verify_events[self.L][1].record()


def e2e_step(r: GpuRound, host, path):
    """The same round through the public API with host buffers: copy the
    round's inputs in from pinned memory, run it, read the accepted tokens."""
    r.inputs.copy_(host["inputs"], non_blocking=True)
    r.step(path)
    host["outputs"].copy_(r.outputs, non_blocking=True)


def e2e_graph_step(r: GpuRound, host, graph):
    """e2e_step with the round's calls replayed from a CUDA graph captured
    from them (the copies stay outside the graph, on the same stream)."""
    r.inputs.copy_(host["inputs"], non_blocking=True)
    graph.replay()
    host["outputs"].copy_(r.outputs, non_blocking=True)


def measure_lookup(w: workloads.Workload, dev, reps: int = 50, min_len: int = 6, max_len: int = 12, k: int = 15):
    """Lookup drafting (stv_lookup_draft) over one history per request of
    the workload, as long as its context (quoted spans planted with p = 0.7).
    L2 is flushed before every timed call (the histories alone would fit in
    L2); CUDA events around each call.  Bytes = 4 per history token."""
    import torch

    import speculative_tree_verify_bit_gb300 as stv

    hs = [torch.as_tensor(h, device=dev) for h in workloads.lookup_histories(w)]
    n = len(hs)
    n_prop = torch.zeros(n, dtype=torch.int32, device=dev)
    prop = torch.zeros((n, k), dtype=torch.int32, device=dev)
    mlen = torch.zeros(n, dtype=torch.int32, device=dev)
    mpos = torch.zeros(n, dtype=torch.int64, device=dev)
    ws = torch.zeros(stv.stv_lookup_workspace_bytes(n), dtype=torch.uint8, device=dev)  # left zero by each call
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    times = []
    for i in range(reps + 3):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        stv.stv_lookup_draft(hs, min_len, max_len, k, n_prop, prop, mlen, mpos, ws)
        b.record()
        torch.cuda.synchronize()
        if i >= 3:
            times.append(a.elapsed_time(b) * 1e3)
    us = statistics.median(times)
    nbytes = 4 * sum(h.numel() for h in hs)
    peak, kind = measured_peak()
    return {"us_per_call": us, "requests": n, "history_tokens": sum(h.numel() for h in hs), "k": k,
            "min_len": min_len, "max_len": max_len, "bytes": nbytes, "gbs": nbytes / (us * 1e-6) / 1e9,
            "frac": nbytes / (us * 1e-6) / 1e9 / peak, "peak_source": kind, "l2": "flushed before each call",
            "proposed": int(n_prop.sum().item())}


def measured_bf16_peak():
    """Dense fp16/bf16 tensor peak (TFLOP/s, burst) from MEASURED_PEAKS.json."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def measure_prefill(dev, n: int = 32768, reps: int = 3, hq: int = 24, hkv: int = 4, path: str = "exact"):
    """Prefill attention (stv_prefill_attn) of an n-token prompt on an empty
    cache, one layer: the prompt's K/V are packed into the 3-bit cache, then
    every token attends causally.  Algorithmic FLOPs = 4 hq D sum_t (t + 1)
    (Q.K^T and P.V over the visible keys); tensor-bound in intent, so the
    fraction is against the measured dense fp16/bf16 peak."""
    import torch

    import speculative_tree_verify_bit_gb300 as stv

    pages = -(-n // 256) + 1
    table = torch.as_tensor(np.random.default_rng(77).permutation(pages).astype(np.int32), device=dev)
    k, v = workloads.kv_rows(4242, n, hkv, device=dev)
    q = workloads.q_rows(4243, 1, n, hq, device=dev)[0].contiguous()
    layer = stv.LayerCache.empty(pages, hkv, device=dev)
    shape = stv.make_shape(hq, hkv)
    stv.stv_kv_append_pack(shape, layer, [stv.Seq(table, 0)], k.contiguous(), v.contiguous(),
                           torch.zeros(n, dtype=torch.int32, device=dev),
                           torch.arange(n, dtype=torch.int32, device=dev))
    seq = stv.Seq(table, 0)
    ws = torch.empty(stv.stv_prefill_workspace_bytes(shape, seq, n), dtype=torch.uint8, device=dev)
    o = torch.empty((n, hq, 256), dtype=torch.float16, device=dev)
    stv.stv_prefill_attn(shape, layer, seq, q, n, path, ws, o)  # warm-up
    times = []
    with ClockSampler(torch.cuda.current_device()) as clk:
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            stv.stv_prefill_attn(shape, layer, seq, q, n, path, ws, o)
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    flops = 4.0 * hq * 256 * (n * (n + 1) / 2)
    peak, kind = measured_bf16_peak()
    tflops = flops / (ms * 1e-3) / 1e12
    kernel = ("prefill_tc (persistent, one launch)" if path == "exact"
              else "verify_i8 over 64-chunk launches + split_combine")
    return {"prompt_tokens": n, "layers": 1, "path": path, "kernel": kernel, "ms_per_call": ms,
            "tokens_per_s": n / (ms * 1e-3), "bound": "tensor", "tflops": tflops, "peak_tflops": peak,
            "frac": tflops / peak, "peak_source": kind, "clocks": clk.summary()}


def measure_ctx_sweep(dev, ctxs=(0, 1024, 4096, 8192, 16384, 32768, 65536, 131072, 262144), reps: int = 15,
                      hq: int = 24, hkv: int = 4, t: int = 16):
    """verify_attn and split_combine launch times against context length: one
    sequence, one layer, T = 16 (a chain tree), exact path; L2 flushed before
    each timed pair, each launch on its own (so each pays its whole fixed
    part: launch, set-up, pipeline fill, epilogue).  A least-squares line
    through the points from 16K keys up, where the split plan gives about one
    work unit per SM, separates the fixed part from the cost per key."""
    import torch

    import speculative_tree_verify_bit_gb300 as stv

    shape = stv.make_shape(hq, hkv)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    points = []
    for ctx in ctxs:
        pages = workloads.pages_needed(ctx, t) + 1
        table = torch.as_tensor(np.random.default_rng(5).permutation(pages).astype(np.int32), device=dev)
        layer = stv.LayerCache.empty(pages, hkv, device=dev)
        k, v = workloads.kv_rows(77, ctx + t, hkv, device=dev)
        stv.stv_kv_append_pack(shape, layer, [stv.Seq(table, 0)], k.contiguous(), v.contiguous(),
                               torch.zeros(ctx + t, dtype=torch.int32, device=dev),
                               torch.arange(ctx + t, dtype=torch.int32, device=dev))
        seqs = [stv.Seq(table, ctx)]
        q = workloads.q_rows(78, 1, t, hq, device=dev).contiguous()
        parent = torch.as_tensor(workloads.chain_tree(t)[None], device=dev)
        ws = torch.empty(stv.stv_verify_workspace_bytes(shape, seqs, t), dtype=torch.uint8, device=dev)
        o = torch.empty((1, t, hq, 256), dtype=torch.float16, device=dev)
        for _ in range(3):
            stv.stv_verify_attn(shape, layer, seqs, q, parent, t, "exact", ws)
            stv.stv_split_combine(shape, seqs, t, ws, o)
        tv, tc = [], []
        for _ in range(reps):
            flush.fill_(1)
            a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            a.record()
            stv.stv_verify_attn(shape, layer, seqs, q, parent, t, "exact", ws)
            b.record()
            stv.stv_split_combine(shape, seqs, t, ws, o)
            c.record()
            torch.cuda.synchronize()
            tv.append(a.elapsed_time(b) * 1e3)
            tc.append(b.elapsed_time(c) * 1e3)
        points.append({"ctx": ctx, "verify_us": statistics.median(tv), "combine_us": statistics.median(tc)})
        del layer, ws
        torch.cuda.empty_cache()
    xs = [p["ctx"] for p in points if p["ctx"] >= 16384]
    ys = [p["verify_us"] for p in points if p["ctx"] >= 16384]
    fit = None
    if len(xs) >= 2:
        slope, icpt = np.polyfit(np.asarray(xs, float), np.asarray(ys, float), 1)
        fit = {"fixed_us": float(icpt), "us_per_1k_keys": float(slope * 1024), "from_ctx": 16384}
    return {"points": points, "fit": fit, "l2": "flushed before each timed launch pair", "path": "exact",
            "t_nodes": t, "hq": hq, "hkv": hkv}


def measure_format(w: workloads.Workload, p_accept: float, dev, kind: str, path: str = "exact", reps: int = 10):
    """The same round over another cache format (the int4 per-token-head
    cache, or the K 4 / V 2-bit cache): two layers resident, eager rounds with
    events around each verify launch; the layers alternate, so a launch does
    not find its cache in L2 (one layer's cache is larger than L2 at 262K)."""
    import torch

    import speculative_tree_verify_bit_gb300 as stv

    group = KV_FORMATS[kind][0]
    r = GpuRound(w, p_accept, dev, layers=2, group=group,
                 kv_format=stv.STV_KV_K4V2 if kind == "k4v2" else stv.STV_KV_BY_GROUP)
    for _ in range(3):
        r.step(path)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(r.L)]
    times, rounds = [], []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        r.step(path, verify_events=ev)
        b.record()
        torch.cuda.synchronize()
        times += [x.elapsed_time(y) for x, y in ev]
        rounds.append(a.elapsed_time(b))
    st = int(r.status.item())
    v_us = statistics.median(times) * 1e3
    vbytes = verify_kernel_bytes(w.ctx, w.t_nodes, w.hq, w.hkv, kind)
    peak, pkind = measured_peak()
    tf, _ = measured_bf16_peak()
    vflops = verify_kernel_flops(w.ctx, w.t_nodes, w.hq)
    gbs = vbytes / (v_us * 1e-6) / 1e9
    out = {"workload": w.name, "kv_format": kind, "group": group, "path": path, "verify_us_per_launch": v_us,
           "eager_us_per_layer_round": statistics.median(rounds) * 1e3 / r.L, "bound": "hbm",
           "algorithmic_bytes_per_launch": vbytes, "achieved_gbs": gbs, "peak_gbs": peak, "frac": gbs / peak,
           "tensor_frac": vflops / (v_us * 1e-6) / 1e12 / tf, "peak_source": pkind, "dev_status": st}
    del r
    torch.cuda.empty_cache()
    return out


def max_over_ranks(values, dist=None, device="cpu"):
    """Each value's maximum over all ranks (the slowest replica sets the
    job's time); unchanged on one process."""
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def us_per_layer_round(round_ms: float, layers: int, world: int) -> float:
    """Whole-job value: N replicas each complete `layers` layer-rounds in the
    slowest rank's round time, so the job does N x layers of them."""
    return round_ms * 1e3 / (layers * world)


def graph_event():
    """An event record node inside a CUDA graph (timing-capable), if this
    PyTorch can make one."""
    import torch

    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None


def time_round(r: GpuRound, path: str, steps: int, warmup: int, barrier, dev):
    """The round (L x append/verify/combine, accept, commit) captured once in
    a CUDA graph; `steps` replays timed with CUDA events, clocks sampled
    meanwhile.  The verify launch times come from a second capture of the
    same round with event record nodes around each layer's verify launch
    (kept out of the timed graph: an event node between two launches
    replaces their programmatic dependency with a full one).
    Returns the replay times (ms), the verify launch times (ms) and the clock
    summary."""
    import torch

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warmup):
            r.step(path)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ev = [[graph_event(), graph_event()] for _ in range(r.L + 1)]  # each verify, then accept + commit
    if any(e is None for pair in ev for e in pair):
        ev = None
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        r.step(path)
    graph_ev = None
    if ev is not None:
        graph_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_ev):
            r.step(path, verify_events=ev)
    for _ in range(warmup):
        graph.replay()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    barrier()
    with ClockSampler(dev.index) as clk:
        marks[0].record()
        for k in range(steps):
            graph.replay()
            marks[k + 1].record()
        barrier()
    round_ms = [marks[k].elapsed_time(marks[k + 1]) for k in range(steps)]
    # per-launch verify time: the event nodes of a few replays of the second graph
    verify_ms = []
    r.accept_commit_ms = []
    if graph_ev is not None:
        graph_ev.replay()  # its first replay uploads the graph
        torch.cuda.synchronize()
    for _ in range(5):
        if graph_ev is not None:
            graph_ev.replay()
            torch.cuda.synchronize()
            verify_ms += [a.elapsed_time(b) for a, b in ev[:r.L]]
            r.accept_commit_ms.append(ev[r.L][0].elapsed_time(ev[r.L][1]))
        else:  # no event nodes: the same launches, eagerly, with events around verify
            ev_eager = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(r.L)]
            r.step(path, verify_events=ev_eager)
            torch.cuda.synchronize()
            verify_ms += [a.elapsed_time(b) for a, b in ev_eager]
    del graph, graph_ev
    return round_ms, verify_ms, clk.summary()


def config_line(w: workloads.Workload, path: str, p_accept: float, kv_format: str, round_ms, verify_ms, clocks,
                layers: int, status: int) -> dict:
    """One workload's figures: round time per layer-round, the verify
    launch, its algorithmic bytes and FLOPs and their fractions of the
    measured HBM and dense fp16/bf16 tensor peaks."""
    us_lr = statistics.median(round_ms) * 1e3 / layers
    v_us = statistics.mean(verify_ms) * 1e3
    vbytes = verify_kernel_bytes(w.ctx, w.t_nodes, w.hq, w.hkv, kv_format)
    vflops = verify_kernel_flops(w.ctx, w.t_nodes, w.hq)
    hbm, _ = measured_peak()
    tf, _ = measured_bf16_peak()
    gbs = vbytes / (v_us * 1e-6) / 1e9
    tflops = vflops / (v_us * 1e-6) / 1e12
    return {"workload": w.name, "ctx": list(w.ctx), "path": path, "p_accept": p_accept, "kv_format": kv_format,
            "us_per_layer_round": us_lr, "verify_us_per_launch": v_us, "algorithmic_bytes_per_launch": vbytes,
            "algorithmic_flops_per_launch": vflops, "hbm_gbs": gbs, "hbm_frac": gbs / hbm, "tflops": tflops,
            "tensor_frac": tflops / tf, "clocks": clocks, "dev_status": status}


def run_gpu(args, rank, world):
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = workloads.WORKLOADS[args.workload]
    p_accept = default_p_accept(args, w)
    r = GpuRound(w, p_accept, dev, layers=args.layers, fuse_append=args.fuse_append,
                 group=KV_FORMATS[args.kv_format][0], kv_format=2 if args.kv_format == "k4v2" else 0,
                 one_launch=args.one_launch)
    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    round_ms, verify_ms, clocks = time_round(r, args.path, args.steps, args.warmup, barrier, dev)
    ac_us = statistics.median(r.accept_commit_ms) * 1e3 if r.accept_commit_ms else None
    st = int(r.status.item())

    # e2e: the round's inputs copied in from pinned host memory (one buffer:
    # Q and the tree K/V rows of every layer, the trees) and its results read
    # back (commit counts, accepted ids), both inside the timed region.  The
    # round's public calls run as a server runs them: captured once into a
    # CUDA graph, replayed each step between the two copies.  The same steps
    # with the calls made eagerly from Python are reported beside it (at
    # short contexts the host's per-call cost, not the GPU, sets that one).
    host = {"inputs": r.inputs.cpu().pin_memory(), "outputs": torch.zeros_like(r.outputs, device="cpu").pin_memory()}
    h2d = host["inputs"].numel()
    d2h = host["outputs"].numel()

    def timed_e2e(one_step):
        for _ in range(2):
            one_step()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            one_step()
        e1.record()
        barrier()
        return e0.elapsed_time(e1)

    e2e_eager_ms = timed_e2e(lambda: e2e_step(r, host, args.path))
    round_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(round_graph):
        r.step(args.path)
    e2e_ms = timed_e2e(lambda: e2e_graph_step(r, host, round_graph))
    del round_graph

    med_ms = statistics.median(round_ms)  # a round = one graph replay
    extra = rank == 0 and not args.no_next_rows
    configs = {}
    if extra and args.workload == "long262k" and args.kv_format == "bit3" and not args.fuse_append:
        # The rest of the metric: the other path and acceptance probabilities
        # on the same resident 262K cache, then the 32K and ragged workloads.
        # Fewer replays each: these are reported beside the headline.
        n = max(5, min(args.steps, 20))
        other = "int8" if args.path == "exact" else "exact"
        rm, vm, ck = time_round(r, other, n, 3, barrier, dev)
        configs[f"long262k/{other}/p{p_accept:g}"] = config_line(w, other, p_accept, "bit3", rm, vm, ck, r.L,
                                                                  int(r.status.item()))
        for pa in w.p_accept:
            if pa == p_accept:
                continue
            r.set_trees(pa)
            rm, vm, ck = time_round(r, args.path, n, 3, barrier, dev)
            configs[f"long262k/{args.path}/p{pa:g}"] = config_line(w, args.path, pa, "bit3", rm, vm, ck, r.L,
                                                                   int(r.status.item()))
        r.set_trees(p_accept)
    lookup = measure_lookup(w, dev) if extra else None
    prefill = measure_prefill(dev) if extra else None
    prefill_i8 = measure_prefill(dev, reps=1, path="int8") if extra else None
    int4 = measure_format(w, p_accept, dev, "int4", args.path) if extra and args.kv_format == "bit3" else None
    k4v2 = measure_format(w, p_accept, dev, "k4v2") if extra and args.kv_format == "bit3" else None
    if configs:
        del r
        torch.cuda.empty_cache()
        for name in ("tree32k", "ragged"):
            w2 = workloads.WORKLOADS[name]
            pa2 = w2.p_accept[0]
            r2 = GpuRound(w2, pa2, dev, one_launch=args.one_launch)
            rm, vm, ck = time_round(r2, args.path, n, 3, barrier, dev)
            configs[f"{name}/{args.path}/p{pa2:g}"] = config_line(w2, args.path, pa2, "bit3", rm, vm, ck, r2.L,
                                                                  int(r2.status.item()))
            del r2
            torch.cuda.empty_cache()
    med_ms, e2e_ms, e2e_eager_ms = max_over_ranks([med_ms, e2e_ms, e2e_eager_ms], dist, dev)
    L = args.layers or w.layers
    layer_rounds = args.steps * L * world
    us_per_lr = us_per_layer_round(med_ms, L, world)
    e2e_us = e2e_ms * 1e3 / layer_rounds
    e2e_eager_us = e2e_eager_ms * 1e3 / layer_rounds
    bytes_lr = algorithmic_bytes_per_layer_round(w.ctx, w.t_nodes, w.hq, w.hkv, args.kv_format)
    vbytes = verify_kernel_bytes(w.ctx, w.t_nodes, w.hq, w.hkv, args.kv_format)
    vflops = verify_kernel_flops(w.ctx, w.t_nodes, w.hq)
    v_us = statistics.mean(verify_ms) * 1e3
    peak, peak_kind = measured_peak()
    achieved = vbytes / (v_us * 1e-6) / 1e9
    traffic = load_traffic(args.workload, args.path, args.kv_format)
    return dict(rank=rank, us_per_lr=us_per_lr, e2e_us=e2e_us, e2e_eager_us=e2e_eager_us, bytes_lr=bytes_lr, v_us=v_us, vbytes=vbytes,
                vflops=vflops, peak=peak, peak_kind=peak_kind, achieved=achieved, clocks=clocks, status=st,
                h2d=h2d, d2h=d2h, launches=launches_per_step(args, w) * args.steps, p_accept=p_accept,
                traffic=traffic, round_gbs=bytes_lr / (us_per_lr * 1e-6) / 1e9 / world, lookup=lookup,
                prefill=prefill, prefill_i8=prefill_i8, int4=int4, k4v2=k4v2, configs=configs, ac_us=ac_us)


KERNEL_SOURCES = {  # the files a verify launch's code comes from, per path and cache format
    "verify_tc": ("csrc/verify_tc.cu", "csrc/tc_util.cuh", "csrc/stv_device.cuh", "csrc/combine.cuh"),
    "verify_i8": ("csrc/verify_i8.cu", "csrc/tc_util.cuh", "csrc/stv_device.cuh"),
}


def verify_kernel_name(path: str, kv_format: str) -> str:
    return "verify_i8" if path == "int8" and kv_format == "bit3" else "verify_tc"


def kernel_sources_sha256(kernel: str) -> str:
    import hashlib

    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(ROOT, "speculative_tree_verify_bit_gb300", f), "rb").read())
    return h.hexdigest()


def load_traffic(workload, path, kv_format="bit3"):
    """DRAM bytes per verify launch from the committed ncu summary, or None
    when there is none for this workload or the kernel's sources have changed
    since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        key = f"{workload}/{path}" + ("" if kv_format == "bit3" else f"/{kv_format}")
        e = d.get("launches", {}).get(key)
        if not e or e.get("sources_sha256") != kernel_sources_sha256(verify_kernel_name(path, kv_format)):
            return None
        return e.get("dram_bytes")
    except Exception:
        return None


# --------------------------------------------------------------------------
# CPU baseline: the fp64 oracle on the host cores, bounded sample
# --------------------------------------------------------------------------

def oracle_sample(w: workloads.Workload, n_rows: int, threads: int, kv_format: str = "bit3"):
    """Time the oracle on n_rows (node, Q head) rows of layer 0 over the full
    context; scale to microseconds per layer-round (all T * hq rows of every
    sequence).  The oracle's own cache is packed first (set-up, untimed)."""
    import torch

    import oracle

    T, hq, hkv = w.t_nodes, w.hq, w.hkv
    pool_pages, tables = workloads.page_tables_for(w)
    cache = oracle.Cache(hkv, pool_pages, bits=4 if kv_format == "int4" else 3, kind=kv_format)
    seed = workloads.layer_seed(w, 0)
    # the sample covers the largest sequence (the long-context share dominates)
    s = int(np.argmax(w.ctx))
    c = w.ctx[s]
    k, v = workloads.kv_rows(seed + 7919 * s, c + T, hkv, device="cpu" if not torch.cuda.is_available() else "cuda")
    k, v = k.cpu().numpy(), v.cpu().numpy()
    oracle.kv_append(cache, [tables[i] if i == s else np.zeros(0, np.int32) for i in range(len(tables))], k, v,
                     np.full(c + T, s, np.int32), np.arange(c + T, dtype=np.int32))
    q = workloads.q_rows(seed, w.n_seqs, T, hq, device="cpu").numpy()
    rt = workloads.round_trees(w)
    rows = [(s, n % T, (n * 7) % hq) for n in range(n_rows)]
    ctx = [c if i == s else 0 for i in range(w.n_seqs)]
    tabs = [tables[i] if i == s else np.zeros(1, np.int32) for i in range(len(tables))]
    t0 = time.perf_counter()
    oracle.attention(cache, tabs, ctx, q, rt.parent, hq, "exact", rows=rows, n_threads=threads)
    dt = time.perf_counter() - t0
    keys_sampled = n_rows * (c + T)
    keys_all = sum(cc + T for cc in w.ctx) * T * hq
    us_per_lr = dt * 1e6 * keys_all / keys_sampled
    sample = (f"oracle attention (fp64, exact path, {kv_format} cache) for {n_rows} of {T * hq * w.n_seqs} (node, Q head) rows of "
              f"layer 0 over the {c}-key context of sequence {s}, scaled by visible keys to one full layer-round")
    return us_per_lr, dt, sample


def arm_config(args, w: workloads.Workload, p_accept: float, world: int) -> dict:
    """The workload both arms (the GPU path and the oracle) report."""
    return {"workload": w.name, "ctx": list(w.ctx), "t_nodes": w.t_nodes, "layers": args.layers or w.layers,
            "hq": w.hq, "hkv": w.hkv, "head_dim": 256, "path": args.path, "p_accept": p_accept,
            "l2": "inputs larger than L2 (16 layers of packed KV)", "parallelism": f"replicas{world}",
            "timing": "median over steps of one CUDA-graph replay of the round, CUDA events",
            "append": ("one launch per layer: append, verify and merge" if args.one_launch and args.path == "exact"
                       else "fused into verify" if args.fuse_append else "separate launch"),
            "kv_format": {"bit3": "3-bit codes, fp16 scale per 32-group",
                          "int4": "int4 codes, fp16 scale per token and KV head",
                          "k4v2": "K 4-bit / V 2-bit codes, fp16 scale per 32-group"}[args.kv_format]}


def default_p_accept(args, w: workloads.Workload) -> float:
    return args.p_accept if args.p_accept is not None else w.p_accept[-1 if args.workload == "long262k" else 0]


def run_reference(args):
    w = workloads.WORKLOADS[args.workload]
    threads = os.cpu_count() or 1
    vals = []
    for _ in range(args.warmup):
        pass  # the oracle has no warm state; warm-up steps are not repeated
    n_rows = args.oracle_rows
    for _ in range(max(1, args.steps)):
        v, dt, sample = oracle_sample(w, n_rows, threads, args.kv_format)
        vals.append(v)
        if dt > 60:
            break
    val = statistics.median(vals)
    line = {
        "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus, "steps": len(vals),
        "warmup": args.warmup, "ms_per_step": val * w.layers / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": arm_config(args, w, default_p_accept(args, w), 1),
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="long262k", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--path", default="exact", choices=["exact", "int8"])
    ap.add_argument("--p-accept", type=float, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--oracle-rows", type=int, default=32)
    ap.add_argument("--layers", type=int, default=None, help="fewer layers (profiling captures only)")
    ap.add_argument("--fuse-append", action="store_true",
                    help="append the tree rows inside the verify launch (stv_append_verify_attn) instead of "
                         "with their own launch")
    ap.add_argument("--one-launch", action="store_true",
                    help="exact path: each layer's append, verify and merge in one cooperative launch "
                         "(stv_append_verify_combine) instead of three")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kv-format", default="bit3", choices=sorted(KV_FORMATS),
                    help="cache format: the 3-bit cache (default), the int4 per-token-head cache or the "
                         "K 4 / V 2-bit cache")
    ap.add_argument("--prefill-only", type=int, default=None, metavar="N",
                    help="time only prefill attention of an N-token prompt (on --path, --steps calls) and print its JSON "
                         "(profiling captures of the prefill kernel)")
    ap.add_argument("--ctx-sweep", action="store_true",
                    help="time verify_attn and split_combine launches alone against context length, one "
                         "layer, and print their JSON (the fixed part of a launch and the cost per key)")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the other configs, lookup, prefill and other-format measurements "
                         "(profiling captures)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.fuse_append and args.kv_format != "bit3":
        ap.error("--fuse-append packs the 3-bit cache only")
    if args.one_launch and (args.kv_format != "bit3" or args.fuse_append):
        ap.error("--one-launch runs the 3-bit cache, without --fuse-append")
    if args.path == "int8" and args.kv_format == "k4v2":
        ap.error("the K 4 / V 2-bit cache runs the exact path only")

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    if args.ctx_sweep:
        if rank == 0:
            print(json.dumps({"ctx_sweep": measure_ctx_sweep("cuda")}), flush=True)
        return
    if args.prefill_only:
        if rank == 0:
            print(json.dumps({"prefill_attn": measure_prefill("cuda", n=args.prefill_only, reps=args.steps,
                                                              path=args.path)}), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    res = run_gpu(args, rank, world)
    if rank != 0:
        return
    w = workloads.WORKLOADS[args.workload]
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        threads = os.cpu_count() or 1
        v, dt, sample = oracle_sample(w, args.oracle_rows, threads, args.kv_format)
        v1, dt1, sample1 = oracle_sample(w, max(1, args.oracle_rows // 8), 1, args.kv_format)
        cpu = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
               "value_1thread": v1, "sample_1thread": sample1}
    tf_peak, tf_kind = measured_bf16_peak()
    tflops = res["vflops"] / (res["v_us"] * 1e-6) / 1e12
    line = {
        "metric": METRIC, "value": res["us_per_lr"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["us_per_lr"] * (args.layers or w.layers) * world / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": arm_config(args, w, res["p_accept"], world),
        "gbs_per_layer_round": res["round_gbs"],
        "bytes_per_layer_round": res["bytes_lr"],
        "verify_us_per_launch": res["v_us"],
        "accept_commit_us_per_round": res.get("ac_us"),
        # The verify launch's arithmetic intensity (FLOPs per algorithmic byte)
        # is above the GPU's ridge point, so its roofline is the dense fp16
        # tensor peak; the HBM figures are beside it.
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": tf_peak, "unit": "TFLOP/s",
                     "frac": tflops / tf_peak, "traffic": res["traffic"], "kernel": "verify_attn",
                     "algorithmic_flops_per_launch": res["vflops"], "algorithmic_bytes_per_launch": res["vbytes"],
                     "arithmetic_intensity": res["vflops"] / res["vbytes"], "ridge": tf_peak * 1e3 / res["peak"],
                     "peak_source": f"{tf_kind} dense bf16 burst (fp16 runs at the same rate)",
                     "hbm_achieved_gbs": res["achieved"], "hbm_peak_gbs": res["peak"],
                     "hbm_frac": res["achieved"] / res["peak"], "hbm_peak_source": res["peak_kind"]},
        "cpu_baseline": cpu,
        "e2e": {"value": res["e2e_us"], "unit": UNIT, "h2d_bytes_per_step": res["h2d"],
                "d2h_bytes_per_step": res["d2h"],
                "calls": "the round's public calls captured once in a CUDA graph, replayed each step "
                         "between the host-to-device and device-to-host copies",
                "eager_value": res["e2e_eager_us"]},
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "dev_status": res["status"],
        "configs": res["configs"],
        "next_rows": {"lookup_draft": res.get("lookup"), "prefill_attn": res.get("prefill"),
                      "prefill_attn_int8": res.get("prefill_i8"),
                      "int4_cache_verify": res.get("int4"), "k4v2_cache_verify": res.get("k4v2")},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
