#!/usr/bin/env python
"""Decode-attention benchmark of the OSCAR INT2 KV-cache path on GB300.

One step = the attention of one decode token for every layer of the model:
per layer, q·R_K + INT2 history (64-token units taken dynamically by the
history CTAs) + BF16 sink/recent partials in one launch
(oscar_decode_attention_fused), then the online-softmax merge with R_V^T
(oscar_merge); for workloads that demote every step, the demotion of the
token leaving the recent window runs inside the same decode launch.
Steps are captured in a CUDA graph and timed with CUDA events.

Prints one JSON line (rank 0).  Default workload: Qwen3-8B shape at 100,000
tokens of context, batch 1, 36 layers.  `--impl reference` times the CPU
oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oscar_synthetic as syn  # noqa: E402

METRIC = "INT2-history decode-attn tokens/s and HBM GB/s (% of roofline) at 100K ctx"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
D = 128


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["oscar", "reference"], default="oscar")
    ap.add_argument("--workload", default="qwen3_8b_100k", choices=sorted(syn.WORKLOADS))
    ap.add_argument("--splits", type=int, default=0, help="history splits per request (0 = library suggestion)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-bf16", action="store_true", help="skip the all-BF16 cache comparison")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU seconds of the oracle sample")
    ap.add_argument("--layers", type=int, default=0, help="profiling aid: run only this many layers (0 = all)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="launch every kernel after the previous one completes (no programmatic dependent launch)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the batch-32 target configuration and the 32K per-step demotion measurements")
    ap.add_argument("--path", choices=["fused", "shared_prefix"], default="fused",
                    help="the step's attention call: oscar_decode_attention_fused (default) or, for workloads with "
                         "a shared prefix, oscar_rotate_q + oscar_decode_attention_shared_prefix")
    ap.add_argument("--bf16-budget", action="store_true",
                    help="run the all-BF16 comparison at this workload's cache footprint: the largest batch of "
                         "its requests whose BF16 cache (shared-prefix pages once) fits in the HBM that the "
                         "INT2 + BF16-window cache takes; report job-level tokens/s of both")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers --

def workload_text(w: syn.Workload) -> str:
    ctx = f"contexts U{{{w.ragged[0]}..{w.ragged[1]}}}" if w.ragged else f"context {w.context}"
    extra = f", {w.shared_prefix}-token shared prefix" if w.shared_prefix else ""
    dem = ", one demotion per request/layer/kv head per step (inside the decode launch)" if w.demote_per_step else ""
    return (f"{w.name}: {w.layers} layers, {w.n_q_heads} q / {w.n_kv_heads} kv heads, head_dim {w.head_dim}, "
            f"batch {w.batch}, {ctx} ({w.sink} BF16 sink + INT2 history + {w.recent} BF16 recent){extra}, "
            f"page {w.page_size}, group {w.group}{dem}")


def bytes_per_step(w: syn.Workload, seq, hist_end) -> dict:
    """Algorithmic bytes of one step: INT2 codes + scale/zero of the history, BF16 windows, q and out."""
    per_tok_int2 = w.n_kv_heads * (2 * w.head_dim // 4 + 4 * 2 * (w.head_dim // w.group))
    per_tok_bf16 = w.n_kv_heads * 2 * w.head_dim * 2
    hist = sum(max(0, int(h) - w.sink) for h in hist_end)
    bf = sum(int(t) - max(0, int(h) - w.sink) for t, h in zip(seq, hist_end))
    qo = w.batch * w.n_q_heads * w.head_dim * 2 * 2
    per_layer = hist * per_tok_int2 + bf * per_tok_bf16 + qo
    return {"int2_per_layer": hist * per_tok_int2, "bf16_per_layer": bf * per_tok_bf16, "qo_per_layer": qo,
            "per_layer": per_layer, "per_step": per_layer * w.layers,
            "bf16_cache_per_step": (sum(seq) * per_tok_bf16 + qo) * w.layers}


def cache_page_bytes(w: syn.Workload) -> tuple:
    """Bytes of one page of the INT2 pool (codes of K and V, scale/zero of both) and of one BF16 page (K and V)."""
    ps, H, D = w.page_size, w.n_kv_heads, w.head_dim
    return ps * H * (2 * D // 4 + 4 * 2 * (D // w.group)), ps * H * D * 2 * 2


def bf16_budget_batch(w: syn.Workload, seq, n_int2_pages: int, n_bf16_pages: int) -> dict:
    """The all-BF16 cache at a fixed HBM budget: the budget is what this workload's mixed cache holds
    (its INT2 pages and BF16 window pages, all layers); the BF16 batch is the largest n >= 1 such
    that requests 0..n-1 fit it with every page in BF16, shared-prefix pages counted once."""
    ps = w.page_size
    int2_page, bf16_page = cache_page_bytes(w)
    budget = n_int2_pages * int2_page + n_bf16_pages * bf16_page
    shared = w.shared_prefix // ps
    pages, n = 0, 0
    for b, t in enumerate(seq):
        n_log = (int(t) + ps - 1) // ps
        need = n_log - (min(shared, n_log) if b > 0 else 0)
        if n >= 1 and (pages + need) * bf16_page > budget:
            break
        pages += need
        n += 1
    return {"batch": n, "budget_bytes": budget * w.layers, "bf16_cache_bytes": pages * bf16_page * w.layers}


def bf16_cache_table(w: syn.Workload, seq, max_pages: int) -> tuple:
    """Page table [n, max_pages] of an all-BF16 cache for requests with contexts `seq`; logical pages
    below the shared prefix map to request 0's pages, the rest get their own; -1 past each context.
    Returns (table, number of physical pages)."""
    ps = w.page_size
    shared = w.shared_prefix // ps
    table = -np.ones((len(seq), max_pages), dtype=np.int32)
    n = 0
    for b, t in enumerate(seq):
        for lp in range((int(t) + ps - 1) // ps):
            if b > 0 and lp < shared:
                table[b, lp] = table[0, lp]
            else:
                table[b, lp] = n
                n += 1
    return table, n


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": d.get("bf16_tflops"), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS, "source": "fallback"}


def stored_traffic(kernel: str, workload: str):
    """dram read+write bytes per launch from a committed ncu capture, if the kernel source is unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel, {}).get(workload)
    if not e:
        return None
    if e.get("source_sha256") != source_hash(kernel):
        return None
    return e.get("bytes_per_launch")


# the sources each measured kernel is compiled from (its translation unit and the headers it includes)
KERNEL_SOURCES = {
    "decode_attention": ["attn_int2_mma.cu", "oscar_internal.cuh", "ptx.cuh", "quant.cuh", "merge_math.cuh",
                         "tma.cuh"],
    "bulk_demotion": ["demote_tc.cu", "oscar_internal.cuh", "ptx.cuh", "tma.cuh"],
}


def source_hash(kernel: str) -> str:
    """sha256 over the kernel's source files; a stored ncu figure counts only while it matches."""
    h = hashlib.sha256()
    cs = os.path.join(ROOT, "bit_kv_cache_oscar_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(cs, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    h.update(open(os.path.join(ROOT, "include", "oscar.h"), "rb").read())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    @staticmethod
    def max_sm_mhz(index: int):
        """The GPU's maximum SM clock (MHz) from nvidia-smi, or None."""
        try:
            out = subprocess.run(["nvidia-smi", f"--id={index}", "--query-gpu=clocks.max.sm",
                                  "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20)
            return float(out.stdout.strip().splitlines()[0])
        except (OSError, ValueError, IndexError, subprocess.TimeoutExpired):
            return None

    def summary(self) -> dict:
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ GPU: setup ----

class Model:
    """Caches, rotations and buffers of every layer for one batch (device memory)."""

    def __init__(self, w: syn.Workload, device, n_splits: int, with_bf16_cache: bool, bf16_budget: bool = False,
                 codebook: bool = False):
        import torch
        from bit_kv_cache_oscar_gb300 import binding as ob
        from bit_kv_cache_oscar_gb300 import calibrate

        self.w, self.dev = w, device
        L = self.L = ob.Layout(w.n_kv_heads, w.gqa, w.page_size, w.group, w.sink, w.recent)
        if codebook:
            # a non-uniform (Lloyd-Max) codebook designed from layer 0's rotated calibration rows
            prof = syn.channel_profile(w.seed, 0, w.n_kv_heads)
            qc, kc, vc = syn.calibration_set(w.seed, 0, w.gqa, prof, device=device)
            RK0, RV0 = calibrate.rotations(qc, kc, vc, 1.0 / math.sqrt(w.head_dim))
            lk = calibrate.codebook(torch.bmm(kc.float(), RK0), w.group, 0.96)
            lv = calibrate.codebook(torch.bmm(vc.float(), RV0), w.group, 0.92)
            L = self.L = ob.Layout(w.n_kv_heads, w.gqa, w.page_size, w.group, w.sink, w.recent,
                                   levels_k=lk, levels_v=lv)
            del qc, kc, vc
        self.seq = syn.context_lengths(w)
        self.demote = w.demote_per_step
        # With per-step demotion, attention still reads the demoted token from BF16 this step.
        hist = [min(t, max(w.sink, t - w.recent - (1 if self.demote else 0))) for t in self.seq]
        self.pages = syn.page_layout(w, self.seq, hist_end=hist)
        self.hist_end = self.pages.hist_end
        B, ps = w.batch, w.page_size
        self.sm_scale = 1.0 / math.sqrt(w.head_dim)
        max_hist = max(int(h) - w.sink for h in self.hist_end)
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        self.S = n_splits or ob.oscar_suggest_splits(L, B, max_hist, sms)
        self.int2_table = torch.from_numpy(self.pages.int2_table).to(device)
        self.bf16_table = torch.from_numpy(self.pages.bf16_table).to(device)
        self.seq_len = torch.tensor(self.seq, dtype=torch.int32, device=device)
        self.hist_dev = torch.from_numpy(self.hist_end.astype(np.int32)).to(device)
        self.q_all = torch.empty((w.layers, B, w.n_q_heads, D), dtype=torch.bfloat16, device=device)
        self.out_all = torch.empty((w.layers, B, w.n_q_heads, D), dtype=torch.bfloat16, device=device)
        self.q_rot = torch.empty((B, w.n_q_heads, D), dtype=torch.float32, device=device)
        self.part = ob.Partials.empty(L, B, self.S, device)
        self.tiles = torch.zeros(2 * B, dtype=torch.int32, device=device)   # dynamic history scheduling
        self.layers = []
        self.bf16_full = [] if with_bf16_cache else None
        max_pages = self.pages.int2_table.shape[1]
        self.bf16_fit, self.bf16_batch, n_full_pages = None, B, B * max_pages
        if with_bf16_cache:
            if bf16_budget:
                # the all-BF16 cache of the first requests that fit this cache's HBM footprint
                self.bf16_fit = bf16_budget_batch(w, self.seq, self.pages.n_int2_pages, self.pages.n_bf16_pages)
                self.bf16_batch = self.bf16_fit["batch"]
                table, n_full_pages = bf16_cache_table(w, self.seq[:self.bf16_batch], max_pages)
                self.full_table = torch.from_numpy(table).to(device)
            else:
                self.full_table = torch.arange(B * max_pages, dtype=torch.int32, device=device).view(B, max_pages)
            nb = self.bf16_batch
            # the all-BF16 kernel runs one CTA per split, one resident CTA per SM
            self.S_full = max(1, min(1024, sms // nb))
            self.part_full = ob.Partials.empty(L, nb, self.S_full, device)
            self.out_full = torch.empty((w.layers, nb, w.n_q_heads, D), dtype=torch.bfloat16, device=device)
        # per-step demotion: position hist_end of each request (left the recent window this step)
        self.dem_req = torch.arange(B, dtype=torch.int32, device=device)
        self.dem_pos = torch.from_numpy(self.hist_end.astype(np.int32)).to(device)
        for l in range(w.layers):
            prof = syn.channel_profile(w.seed, l, w.n_kv_heads)
            qc, kc, vc = syn.calibration_set(w.seed, l, w.gqa, prof, device=device)
            RK, RV = calibrate.rotations(qc, kc, vc, self.sm_scale)
            del qc, kc, vc
            i2 = ob.Int2Pool.empty(L, self.pages.n_int2_pages, device)
            bf = ob.Bf16Pool.empty(L, self.pages.n_bf16_pages, device)
            full = ob.Bf16Pool.empty(L, n_full_pages, device) if with_bf16_cache else None
            for b, T in enumerate(self.seq):
                k, v = syn.kv_rows(w.seed, l, b, 0, T, prof, device=device, shared_prefix=w.shared_prefix)
                n_log = (T + ps - 1) // ps
                stage = ob.Bf16Pool.empty(L, n_log, device)
                stage.k.view(-1, w.n_kv_heads, D)[:T] = k
                stage.v.view(-1, w.n_kv_heads, D)[:T] = v
                if full is not None and self.bf16_fit is None:
                    full.k[b * max_pages:b * max_pages + n_log] = stage.k
                    full.v[b * max_pages:b * max_pages + n_log] = stage.v
                elif full is not None and b < self.bf16_batch:
                    # this request's own pages (request 0 also holds the shared prefix)
                    first = 0 if b == 0 else min(w.shared_prefix // ps, n_log)
                    src = torch.arange(first, n_log, device=device)
                    dst = self.full_table[b, first:n_log].long()
                    full.k[dst] = stage.k[src]
                    full.v[dst] = stage.v[src]
                st_table = torch.full((1, max_pages), -1, dtype=torch.int32, device=device)
                st_table[0, :n_log] = torch.arange(n_log, dtype=torch.int32, device=device)
                start = w.sink if b == 0 else max(w.sink, w.shared_prefix)
                stop = int(self.hist_end[b]) + (1 if self.demote else 0)
                if stop > start and not codebook:   # the prefill's history, demoted on the tensor cores
                    rng = torch.tensor([[start], [stop]], dtype=torch.int32, device=device)
                    ob.oscar_demote_range(L, stage, st_table, i2, self.int2_table[b:b + 1].contiguous(), rng[0],
                                          rng[1], RK, RV, 0.96, 0.92)
                elif stop > start:                  # (a non-uniform codebook: the CUDA-core demotion)
                    pos = torch.arange(start, stop, dtype=torch.int32, device=device)
                    ob.oscar_demote(L, stage, st_table, i2, self.int2_table[b:b + 1].contiguous(),
                                    torch.zeros_like(pos), pos, RK, RV, 0.96, 0.92)
                for lp in range(n_log):
                    pg = int(self.pages.bf16_table[b, lp])
                    if pg >= 0:
                        bf.k[pg] = stage.k[lp]
                        bf.v[pg] = stage.v[lp]
                del k, v, stage
            self.q_all[l] = syn.queries(w.seed, l, B, w.gqa, prof, device=device)
            self.layers.append({"RK": RK, "RV": RV, "int2": i2, "bf16": bf})
            if full is not None:
                self.bf16_full.append(full)
        torch.cuda.synchronize()
        assert ob.oscar_get_device_status() == 0

    # One decode step over all layers (the path).  Per layer the BF16 sink/recent half runs on
    # a second stream next to q rotation + the INT2 history half; the merge joins them.
    # Optional events bracket each decode-attention launch.
    def step(self, events=None, demote=None):
        import torch
        from bit_kv_cache_oscar_gb300 import binding as ob
        L, w = self.L, self.w
        cur = torch.cuda.current_stream()
        demote = self.demote if demote is None else demote
        for l, st in enumerate(self.layers):
            if events is not None:
                events[l][0].record()
            # query rotation, the history in 64-token units taken dynamically by the history CTAs,
            # the BF16 window (and the per-step demotion) in one launch; the merge in a second one
            # after the whole grid (programmatic dependent launch).  Starting each request's merge on
            # its clusters' arrival counts (merge_counters=...) measured 3 % slower per step at
            # batch 1; fixed history splits (tile_counters=None) 1.4 % slower.
            ob.oscar_decode_attention_fused(L, self.q_all[l], st["RK"], st["bf16"], self.bf16_table, st["int2"],
                                            self.int2_table, self.seq_len, self.hist_dev, self.sm_scale, self.part,
                                            demote_pos=self.dem_pos if demote else None, R_V=st["RV"],
                                            c_K=0.96, c_V=0.92, tile_counters=self.tiles)
            if events is not None:
                events[l][1].record()
            ob.oscar_merge(L, self.part, st["RV"], self.out_all[l])

    def step_shared_prefix(self, part, prefix_splits: int):
        """The step with the shared prefix read once per kv head for the whole batch: per layer
        oscar_rotate_q, oscar_decode_attention_shared_prefix (prefix slots 0 .. prefix_splits - 1,
        the requests' own histories and windows after them), the per-step demotion through
        oscar_demote when the workload demotes, and oscar_merge."""
        from bit_kv_cache_oscar_gb300 import binding as ob
        L, w = self.L, self.w
        for l, st in enumerate(self.layers):
            ob.oscar_rotate_q(L, self.q_all[l], st["RK"], self.q_rot)
            ob.oscar_decode_attention_shared_prefix(L, self.q_all[l], self.q_rot, st["bf16"], self.bf16_table,
                                                    st["int2"], self.int2_table, self.seq_len, self.hist_dev,
                                                    self.sm_scale, w.shared_prefix, prefix_splits, part,
                                                    tile_counters=self.tiles)
            if self.demote:
                ob.oscar_demote(L, st["bf16"], self.bf16_table, st["int2"], self.int2_table, self.dem_req,
                                self.dem_pos, st["RK"], st["RV"], 0.96, 0.92)
            ob.oscar_merge(L, part, st["RV"], self.out_all[l])

    def step_plain(self):
        """The step through oscar_rotate_q + oscar_decode_attention + oscar_merge (the path a
        non-uniform codebook takes: its INT2 history on the CUDA cores)."""
        from bit_kv_cache_oscar_gb300 import binding as ob
        for l, st in enumerate(self.layers):
            ob.oscar_rotate_q(self.L, self.q_all[l], st["RK"], self.q_rot)
            ob.oscar_decode_attention(self.L, self.q_all[l], self.q_rot, st["bf16"], self.bf16_table, st["int2"],
                                      self.int2_table, self.seq_len, self.hist_dev, self.sm_scale, self.part)
            ob.oscar_merge(self.L, self.part, st["RV"], self.out_all[l])

    def demote_step(self):
        """The per-step demotion alone: one token per request, layer and kv head (K and V)."""
        from bit_kv_cache_oscar_gb300 import binding as ob
        for st in self.layers:
            ob.oscar_demote(self.L, st["bf16"], self.bf16_table, st["int2"], self.int2_table, self.dem_req,
                            self.dem_pos, st["RK"], st["RV"], 0.96, 0.92)

    def step_bf16(self):
        from bit_kv_cache_oscar_gb300 import binding as ob
        nb = self.bf16_batch
        for l, full in enumerate(self.bf16_full):
            ob.oscar_bf16_decode_attention(self.L, self.q_all[l, :nb], full, self.full_table, self.seq_len[:nb],
                                           self.sm_scale, self.part_full)
            ob.oscar_merge(self.L, self.part_full, None, self.out_full[l])

    def launches_per_step(self) -> int:
        # per layer: rotation + INT2 history + BF16 window (+ the demotion), merge
        return self.w.layers * 2


def capture(fn, steps: int = 1):
    import torch
    fn()                                  # eager warm-up (first-launch attribute set-up)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(steps):
            fn()
    torch.cuda.synchronize()
    return g


def max_over_ranks(t: float, dist=None, device="cuda") -> float:
    """The largest of the ranks' values (the slowest rank sets the step time)."""
    if not dist:
        return t
    import torch
    tt = torch.tensor([t], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_throughput(world: int, batch: int, seconds: float, steps: int) -> float:
    """Whole-job tokens/s: every rank decodes `batch` tokens per step (weak scaling)."""
    return world * batch / (seconds / steps)


def time_graph(g, K: int, W: int, dist=None) -> float:
    """Seconds for K replays (after W warm-up replays), barrier + sync on both sides, max over ranks."""
    import torch
    for _ in range(W):
        g.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(K):
        g.replay()
    e.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    return max_over_ranks(s.elapsed_time(e) / 1e3, dist)


# ---------------------------------------------------------- CPU baseline ----

def oracle_sample(w: syn.Workload, target_s: float, device_for_inputs="cpu") -> dict:
    """Time the oracle's fp64 decode attention for the query heads of kv head 0 of layer 0 of
    request 0 (its own demotion of that head's history beforehand, untimed); extrapolate to one
    step (all query heads, all layers, all requests)."""
    import torch
    import oracle

    def bf16_bits(t):
        return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

    oracle.build()
    prof = syn.channel_profile(w.seed, 0, w.n_kv_heads)
    qc, kc, vc = syn.calibration_set(w.seed, 0, w.gqa, prof)
    sm = 1.0 / math.sqrt(w.head_dim)
    q0 = oracle.bf16_to_f64(bf16_bits(qc[0]))
    RK = oracle.rotation_from_covariance(oracle.query_covariance(q0)).astype(np.float32)
    RV = oracle.rotation_from_covariance(oracle.score_weighted_value_covariance(
        q0, oracle.bf16_to_f64(bf16_bits(kc[0])), oracle.bf16_to_f64(bf16_bits(vc[0])), sm)).astype(np.float32)
    seq = syn.context_lengths(w)
    T = seq[0]
    he = min(T, max(w.sink, T - w.recent))
    k, v = syn.kv_rows(w.seed, 0, 0, 0, T, prof)
    kb, vb = bf16_bits(k[:, 0]), bf16_bits(v[:, 0])
    g = w.group
    ck = np.zeros((T, D // 4), np.uint8)
    cv = np.zeros((T, D // 4), np.uint8)
    zk, sk, zv, sv = (np.zeros((T, D // g), np.uint16) for _ in range(4))
    _, ck[w.sink:he], zk[w.sink:he], sk[w.sink:he] = oracle.demote_rows(kb[w.sink:he], RK, g, 0.96)
    _, cv[w.sink:he], zv[w.sink:he], sv[w.sink:he] = oracle.demote_rows(vb[w.sink:he], RV, g, 0.92)
    cache = oracle.HeadCache(kb, vb, ck, cv, zk, sk, zv, sv, w.sink, he, g)
    qb = bf16_bits(syn.queries(w.seed, 0, 1, w.gqa, prof))

    def run(first: int, stride: int, seconds: float):
        # query heads first, first + stride, ... until `seconds` have passed; the oracle's C
        # call releases the GIL, so threads running this side by side use separate cores
        n, t0 = 0, time.perf_counter()
        while True:
            oracle.attend_head(qb[0, (first + n * stride) % w.gqa], RK, RV, cache, sm)
            n += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return n, el

    # one host core, then every core this process may run on (one thread each)
    n1, el1 = run(0, 1, target_s / 2)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    with concurrent.futures.ThreadPoolExecutor(cores) as ex:
        res = list(ex.map(lambda i: run(i, cores, target_s / 2), range(cores)))
    nN = sum(r[0] for r in res)
    elN = max(r[1] for r in res)
    heads_per_step = w.n_q_heads * w.layers * w.batch
    scale = heads_per_step * (sum(seq) / (T * w.batch))      # query-head attentions of T tokens per step
    step_1 = el1 / n1 * scale
    step_s = elN / nN * scale
    return {"value": w.batch / step_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "single_core_value": w.batch / step_1,
            "sample": (f"{nN} fp64 query-head attentions (layer 0, kv head 0, T={T}) in {elN:.1f} s on "
                       f"{cores} host cores, one thread each (one core alone: {n1} in {el1:.1f} s); one step "
                       f"= {heads_per_step} query-head attentions, scaled by per-head time and context length"),
            "seconds": el1 + elN, "step_s": step_s}


def run_reference(args, w, rank):
    if rank != 0:
        return
    vals = []
    per = max(1.0, args.cpu_seconds / max(1, args.steps))
    for _ in range(args.steps):
        vals.append(oracle_sample(w, per))
    v = statistics.median(x["value"] for x in vals)
    cpu = dict(vals[-1])
    cpu["value"] = v
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * w.batch / v,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_text(w)},
            "cpu_baseline": {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample", "single_core_value")},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def bulk_demotion(model, w, args, dist) -> dict:
    """Bulk demotion of one layer's whole history of request 0 ([sink, hist_end), every kv head,
    K and V) from a BF16 staging pool into a scratch INT2 pool, the pool fill of a prefix hit.

    oscar_demote_range (tensor cores): rows/s; the HBM roofline of its algorithmic bytes (per
    row-head and K/V: the 256-byte bf16 row in, 32 bytes of codes and the bf16 scale/zero out);
    the tensor-pipe rate of the MMAs it issues (x . R_hi + x . R_lo: 2 x 2 x 128 x 128 flops per
    row-head and K/V) against the measured bf16 peak.  oscar_demote's CUDA-core fp32 chain over
    the same rows is timed beside it."""
    import torch
    from bit_kv_cache_oscar_gb300 import binding as ob
    L, dev, ps = model.L, model.dev, w.page_size
    T = int(model.seq[0])
    he = int(model.hist_end[0])
    n_log = (T + ps - 1) // ps
    prof = syn.channel_profile(w.seed, 0, w.n_kv_heads)
    k, v = syn.kv_rows(w.seed, 0, 0, 0, T, prof, device=dev)
    stage = ob.Bf16Pool.empty(L, n_log, dev)
    stage.k.view(-1, w.n_kv_heads, D)[:T] = k
    stage.v.view(-1, w.n_kv_heads, D)[:T] = v
    del k, v
    table = torch.arange(n_log, dtype=torch.int32, device=dev).view(1, n_log)
    i2 = ob.Int2Pool.empty(L, n_log, dev)
    st = model.layers[0]
    pb = torch.tensor([w.sink], dtype=torch.int32, device=dev)
    pe = torch.tensor([he], dtype=torch.int32, device=dev)
    reps = max(3, min(args.steps, 20))
    g = capture(lambda: ob.oscar_demote_range(L, stage, table, i2, table, pb, pe, st["RK"], st["RV"], 0.96, 0.92))
    tb = time_graph(g, reps, args.warmup, dist) / reps
    pos = torch.arange(w.sink, he, dtype=torch.int32, device=dev)
    req = torch.zeros_like(pos)
    gl = capture(lambda: ob.oscar_demote(L, stage, table, i2, table, req, pos, st["RK"], st["RV"], 0.96, 0.92))
    tl = time_graph(gl, reps, args.warmup, dist) / reps
    n_rh = (he - w.sink) * w.n_kv_heads
    unit_bytes = 2 * (D * 2 + D // 4 + 2 * 2 * (D // w.group))   # K and V: bf16 row in; codes, scale, zero out
    bytes_launch = n_rh * unit_bytes
    peaks = measured_peaks()
    achieved = bytes_launch / tb / 1e9
    mma_tflops = n_rh * 2 * 2 * 2 * D * D / tb / 1e12
    bf16_peak = peaks.get("bf16_tflops")
    del stage, i2
    return {"rows": he - w.sink, "row_heads": n_rh, "ms": tb * 1e3, "row_heads_per_s": n_rh / tb,
            "kernel": "oscar_demote_range (bulk_demote_kernel: TMA + tcgen05.mma into TMEM + register quantizer)",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "bytes_per_launch": bytes_launch,
                         "bytes_per_row_head": unit_bytes,
                         "traffic": stored_traffic("bulk_demotion", w.name),
                         "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs copy bandwidth)"},
            "tensor": {"achieved": mma_tflops, "unit": "TFLOP/s", "peak": bf16_peak,
                       "frac": (mma_tflops / bf16_peak) if bf16_peak else None,
                       "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)"},
            "cuda_core_fp32_chain": {"ms": tl * 1e3, "row_heads_per_s": n_rh / tl,
                                     "kernel": "oscar_demote (demote_kernel)"}}


# ------------------------------------------------------------------- main ----

def decode_roofline(model, w, bts, args, torch) -> dict:
    """Per-launch roofline of oscar_decode_attention_fused: events captured around every decode
    launch of a KR-step graph (the events split the launch-overlap edges, so a launch is timed
    alone); algorithmic bytes per launch = the hot-path scope's per-layer bytes (INT2 codes and
    scale/zero of the history, BF16 sink + recent, q and out)."""
    KR = min(args.steps, 20)
    evs = [[(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
            for _ in range(w.layers)] for _ in range(KR)]
    gp = capture(lambda: model.step(events=evs[0]))
    gk = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gk):
        for k in range(KR):
            model.step(events=evs[k])
    for _ in range(args.warmup):
        gp.replay()
    torch.cuda.synchronize()
    gk.replay()
    torch.cuda.synchronize()
    durs = [evs[k][l][0].elapsed_time(evs[k][l][1]) / 1e3 for k in range(KR) for l in range(w.layers)]
    dur = statistics.mean(durs)
    peaks = measured_peaks()
    unit_bytes = bts["per_layer"]
    achieved = unit_bytes / dur / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": stored_traffic("decode_attention", w.name),
            "kernel": "oscar_decode_attention_fused (q.R_K + INT2 history split-K in dynamic 64-token units + "
                      "BF16 window, one layer, one launch)",
            "bytes_per_launch": unit_bytes, "launch_us": dur * 1e6,
            "bytes_definition": "INT2 codes + bf16 scale/zero of [sink, hist_end), BF16 K/V of the sink and recent "
                                "window, q and out (bf16), per layer",
            "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs copy bandwidth)"}


def unique_bytes_per_step(w: syn.Workload, bts: dict) -> int:
    """The step's algorithmic bytes with pages shared by several requests (the common prefix held
    once in the page tables) counted once."""
    if not w.shared_prefix or w.batch < 2:
        return bts["per_step"]
    per_tok_int2 = w.n_kv_heads * (2 * w.head_dim // 4 + 4 * 2 * (w.head_dim // w.group))
    per_tok_bf16 = w.n_kv_heads * 2 * w.head_dim * 2
    shared = (w.shared_prefix - w.sink) * per_tok_int2 + w.sink * per_tok_bf16
    return bts["per_step"] - (w.batch - 1) * shared * w.layers


def demotion_overhead(model, args, dist) -> dict:
    """Step time with the per-step demotion (inside the decode launch) against the same step without."""
    g0 = capture(lambda: model.step(demote=False))
    t0 = time_graph(g0, args.steps, args.warmup, dist) / args.steps
    g1 = capture(lambda: model.step(demote=True))
    t1 = time_graph(g1, args.steps, args.warmup, dist) / args.steps
    del g0, g1
    return {"step_ms_without": t0 * 1e3, "step_ms_with": t1 * 1e3, "step_overhead": t1 / t0,
            "rows_per_step": model.w.layers * model.w.batch * model.w.n_kv_heads * 2,
            "bar": "step time with demotion <= 1.02 x without"}


def range_demotion_step(model, args, dist) -> dict:
    """The per-step demotion's rows (one position per request and layer, every kv head, K and V)
    through the tcgen05 range kernel instead: one oscar_demote_range launch per layer over
    [pos, pos + 1) of every request, timed alone."""
    import torch
    from bit_kv_cache_oscar_gb300 import binding as ob
    end = model.dem_pos + 1

    def step():
        for st in model.layers:
            ob.oscar_demote_range(model.L, st["bf16"], model.bf16_table, st["int2"], model.int2_table,
                                  model.dem_pos, end, st["RK"], st["RV"], 0.96, 0.92)
    g = capture(step)
    t = time_graph(g, args.steps, args.warmup, dist) / args.steps
    del g
    return {"us_per_step": t * 1e6, "us_per_layer": t * 1e6 / model.w.layers,
            "kernel": "oscar_demote_range (bulk_demote_kernel: TMA + tcgen05.mma into TMEM), separate launch"}


def prefix_splits(w) -> int:
    """Token splits of the shared-prefix kernel: one CTA per (split, kv head), one wave."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return max(1, sms // w.n_kv_heads)


def cascade_step(model, w, args, dist, world, fused_sec: float) -> dict:
    """The shared prefix read once per kv head for the whole batch: per layer oscar_rotate_q,
    oscar_decode_attention_shared_prefix (tcgen05 prefix kernel over [sink, shared_prefix) in
    prefix_splits slots + the requests' own histories and windows), the per-step demotion through
    oscar_demote when the workload demotes, and oscar_merge."""
    import torch
    from bit_kv_cache_oscar_gb300 import binding as ob
    ps = prefix_splits(w)
    part = ob.Partials.empty(model.L, w.batch, ps + model.S, model.dev)
    g = capture(lambda: model.step_shared_prefix(part, ps))
    t = time_graph(g, args.steps, args.warmup, dist)
    del g, part
    sec = t / args.steps
    return {"value": job_throughput(world, w.batch, t, args.steps), "unit": "tokens/s", "ms_per_step": sec * 1e3,
            "prefix_splits": ps, "suffix_splits": model.S, "shared_prefix_tokens": w.shared_prefix,
            "step_vs_fused": sec / fused_sec,
            "path": "oscar_rotate_q + oscar_decode_attention_shared_prefix + oscar_demote + oscar_merge per layer"}


def codebook_line(args, dist, world, fused_us_per_layer: float) -> dict:
    """The 100K workload's decode with a non-uniform (Lloyd-Max) codebook, two layers: the history
    demoted through oscar_demote with the layout's levels, the step through oscar_rotate_q +
    oscar_decode_attention (INT2 history on the CUDA cores) + oscar_merge."""
    import dataclasses
    import torch
    w = dataclasses.replace(syn.WORKLOADS["qwen3_8b_100k"], layers=2)
    model = Model(w, torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0"))), args.splits,
                  with_bf16_cache=False, codebook=True)
    g = capture(model.step_plain)
    t = time_graph(g, args.steps, args.warmup, dist) / args.steps
    lk, lv = model.L.levels_k, model.L.levels_v
    del g, model
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    us = t * 1e6 / w.layers
    return {"workload": workload_text(w), "levels_k": lk, "levels_v": lv, "us_per_layer": us,
            "uniform_fused_us_per_layer": fused_us_per_layer, "slowdown_vs_uniform": us / fused_us_per_layer,
            "path": "INT2 history on the CUDA cores (attn_simple int2_split_kernel, codebook lookup)"}


def workload_line(w, args, dist, world, bf16_budget: bool) -> dict:
    """tokens/s, step time and HBM roofline of one workload's decode step (and, with bf16_budget, the
    all-BF16 cache at the same HBM footprint); the per-step demotion's overhead when it demotes."""
    import torch
    model = Model(w, torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0"))), args.splits,
                  with_bf16_cache=bf16_budget, bf16_budget=bf16_budget)
    bts = bytes_per_step(w, model.seq, model.hist_end)
    g = capture(lambda: model.step())
    t = time_graph(g, args.steps, args.warmup, dist)
    del g
    peaks = measured_peaks()
    sec = t / args.steps
    uniq = unique_bytes_per_step(w, bts)
    out = {"workload": workload_text(w), "value": job_throughput(world, w.batch, t, args.steps), "unit": "tokens/s",
           "ms_per_step": sec * 1e3, "history_splits": model.S,
           "bytes_per_step": bts["per_step"], "unique_bytes_per_step": uniq,
           "roofline": {"bound": "hbm", "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "achieved_logical": bts["per_step"] / sec / 1e9,
                        "frac_logical": bts["per_step"] / sec / 1e9 / peaks["hbm_gbs"],
                        "achieved_unique": uniq / sec / 1e9, "frac_unique": uniq / sec / 1e9 / peaks["hbm_gbs"],
                        "note": "whole step (decode launch + merge per layer); logical bytes count the shared "
                                "prefix once per request, unique bytes once"}}
    if model.demote:
        out["per_step_demotion"] = demotion_overhead(model, args, dist)
        if w.batch > 1:
            out["per_step_demotion"]["tensor_core_range_kernel"] = range_demotion_step(model, args, dist)
    if w.shared_prefix > 0:
        out["shared_prefix_cascade"] = cascade_step(model, w, args, dist, world, sec)
    if bf16_budget and model.bf16_full is not None:
        gb = capture(model.step_bf16)
        tb = time_graph(gb, args.steps, args.warmup, dist)
        del gb
        nb = model.bf16_batch
        vb = job_throughput(world, nb, tb, args.steps)
        bb = (sum(model.seq[:nb]) * w.n_kv_heads * w.head_dim * 4 + nb * w.n_q_heads * w.head_dim * 4) * w.layers
        out["bf16_cache_fixed_budget"] = {
            "batch": nb, "value": vb, "unit": "tokens/s", "ms_per_step": 1e3 * tb / args.steps,
            "bytes_per_step": bb, "gbs": bb / (tb / args.steps) / 1e9, "fixed_hbm_budget": model.bf16_fit,
            "int2_job_speedup": out["value"] / vb,
            "comparison": "job-level tokens/s of both caches in the same HBM footprint"}
    del model
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def main():
    args = parse_args()
    w = syn.WORKLOADS[args.workload]
    if args.layers:
        import dataclasses
        w = dataclasses.replace(w, layers=args.layers)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, w, rank)

    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from bit_kv_cache_oscar_gb300 import binding as ob
    ob.lib()
    model = Model(w, torch.device("cuda", local), args.splits, with_bf16_cache=not args.no_bf16,
                  bf16_budget=args.bf16_budget)
    torch.cuda.synchronize()
    # The step's kernels read pools, tables and lengths that no kernel of the step writes
    # (the per-step demotion writes positions the step does not read from INT2), so
    # consecutive kernels may overlap.
    ob.oscar_set_launch_overlap(not args.no_overlap)
    bts = bytes_per_step(w, model.seq, model.hist_end)

    # headline: one-step graph replayed K times
    if args.path == "shared_prefix":
        if not w.shared_prefix:
            raise SystemExit("--path shared_prefix needs a workload with a shared prefix")
        ps = prefix_splits(w)
        part_sp = ob.Partials.empty(model.L, w.batch, ps + model.S, model.dev)
        g = capture(lambda: model.step_shared_prefix(part_sp, ps))
    else:
        g = capture(lambda: model.step())
    with ClockSampler(local) as clk:
        t = time_graph(g, args.steps, args.warmup, dist)
    ms_step = 1e3 * t / args.steps
    value = job_throughput(world, w.batch, t, args.steps)
    roof = decode_roofline(model, w, bts, args, torch)

    # e2e: q from pinned host memory -> step -> out to pinned host memory, every step
    q_host = [torch.empty_like(model.q_all, device="cpu").pin_memory() for _ in range(2)]
    for qh in q_host:
        qh.copy_(model.q_all)
    out_host = [torch.empty_like(model.out_all, device="cpu").pin_memory() for _ in range(2)]
    for k in range(args.warmup):
        model.q_all.copy_(q_host[k % 2], non_blocking=True)
        g.replay()
        out_host[k % 2].copy_(model.out_all, non_blocking=True)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for k in range(args.steps):
        model.q_all.copy_(q_host[k % 2], non_blocking=True)
        g.replay()
        out_host[k % 2].copy_(model.out_all, non_blocking=True)
    e.record()
    torch.cuda.synchronize()
    te = max_over_ranks(s.elapsed_time(e) / 1e3, dist)
    e2e = {"value": job_throughput(world, w.batch, te, args.steps), "unit": "tokens/s",
           "h2d_bytes_per_step": model.q_all.numel() * 2, "d2h_bytes_per_step": model.out_all.numel() * 2}

    # demotion (rows a1-a3): the per-step demotion (one token per request, layer and kv head,
    # folded into the decode launch in the workloads that demote every step) timed alone through
    # oscar_demote and as the step's overhead; and a bulk demotion of one layer's whole history
    # (the pool fill of a prefix hit)
    gd = capture(model.demote_step)
    td = time_graph(gd, args.steps, args.warmup, dist) / args.steps
    gs = capture(lambda: model.step(demote=True))
    ts = time_graph(gs, args.steps, args.warmup, dist) / args.steps
    demotion = {"per_step_us": td * 1e6, "rows_per_step": w.layers * w.batch * w.n_kv_heads * 2,
                "step_ms_with_demotion": ts * 1e3, "step_overhead": ts / (t / args.steps)}
    demotion["bulk"] = bulk_demotion(model, w, args, dist)

    bf16 = None
    if model.bf16_full is not None:
        gb = capture(model.step_bf16)
        tb = time_graph(gb, args.steps, args.warmup, dist)
        nb = model.bf16_batch
        vb = job_throughput(world, nb, tb, args.steps)
        bb = bts["bf16_cache_per_step"]
        if model.bf16_fit is not None:     # the first nb requests' caches and q/out
            bb = (sum(model.seq[:nb]) * w.n_kv_heads * w.head_dim * 4
                  + nb * w.n_q_heads * w.head_dim * 4) * w.layers
        bf16 = {"value": vb, "unit": "tokens/s", "ms_per_step": 1e3 * tb / args.steps,
                "bytes_per_step": bb, "int2_speedup": value / vb, "gbs": bb / (tb / args.steps) / 1e9}
        if model.bf16_fit is not None:
            bf16.update({"batch": nb, "fixed_hbm_budget": model.bf16_fit,
                         "comparison": "job-level tokens/s of both caches in the same HBM footprint"})
    assert ob.oscar_get_device_status() == 0
    del g, gd, gs, model
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    # the other single-GPU configurations of the hot path's scope: the batch-32 target (ragged
    # 64K-100K contexts, 16K shared prefix, per-step demotion) with the all-BF16 cache at the same
    # HBM footprint, and the 32K context whose every step demotes
    extra = None
    if not args.no_extra and args.workload == "qwen3_8b_100k" and not args.layers:
        extra = {"target_batch32": workload_line(syn.WORKLOADS["qwen3_8b_b32_ragged"], args, dist, world, True),
                 "ctx32k_per_step_demotion": workload_line(syn.WORKLOADS["qwen3_8b_32k"], args, dist, world, False),
                 "codebook_lloyd_max_100k": codebook_line(args, dist, world, 1e6 * t / args.steps / w.layers)}
        assert ob.oscar_get_device_status() == 0

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = oracle_sample(w, args.cpu_seconds)
        cpu = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample", "single_core_value")}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp32 accumulate, f16 hi+lo split MMA operands", "data": "synthetic",
            "config": {"workload": workload_text(w), "batch": w.batch, "layers": w.layers,
                       "history_splits": model_splits(w, args),
                       "l2": f"inputs larger than L2: {bts['per_step'] / 1e9:.2f} GB read per step, 129 MB L2",
                       "kv_storage": "INT2 history (codes + bf16 scale/zero per group) + BF16 sink/recent",
                       "timing": "CUDA graph of one step, CUDA events, K replays"},
            "hbm_gbs": bts["per_step"] / (t / args.steps) / 1e9 * world,
            "bytes_per_step": bts["per_step"],
            "roofline": roof,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 2 * w.layers * args.steps,
            "clocks": clk.summary(), "bf16_cache": bf16, "demotion": demotion, "other_configs": extra,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def model_splits(w, args) -> int:
    from bit_kv_cache_oscar_gb300 import binding as ob
    import torch
    L = ob.Layout(w.n_kv_heads, w.gqa, w.page_size, w.group, w.sink, w.recent)
    seq = syn.context_lengths(w)
    hist = [min(t, max(w.sink, t - w.recent - (1 if w.demote_per_step else 0))) for t in seq]
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return args.splits or ob.oscar_suggest_splits(L, w.batch, max(hist) - w.sink, sms)


if __name__ == "__main__":
    main()
