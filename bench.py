#!/usr/bin/env python
"""Benchmark of the Q8_0 GQA verify / prompt attention path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

One JSON line on rank 0.  A step is one speculative-verify step on the long-context
workload (24 q heads / 4 kv heads, head_dim 256, context 20,676): for each window length
T in {4, 8}, one attn_verify_append_q8 call appends the T new K/V tokens to the Q8_0 cache
and runs the verify scan over ctx + T keys: the split-context kernel, whose window slice
quantises the new tokens itself, and the log-sum-exp combine.  The two windows are
independent problems (each on its own cache), run back to back on one stream.
`value` is the KV-scan bandwidth of the whole job (Q8_0 K/V bytes read by the verify
calls / time), in GB/s; `per_T` gives the per-call latency of each window length, `cells`
the same figures at contexts 32,768 and 4,096.  The prompt-chunk kernel (12 q heads /
1 kv head, hd256, 2048 queries over a 32768-token int8 context) is timed in the same run
and reported under "prompt" in TFLOP/s.

Timing: steps are captured in CUDA graphs and replayed, so the device time is not hidden
behind Python launch overhead; exactly --warmup untimed and --steps timed steps run (a graph
of up to 64 steps, replayed, plus one graph of the remainder).  Every step reads a different
cache of a ring whose total size is above 4x the L2, so K/V bytes come from HBM.  The `e2e`
figure instead goes through the C ABI's host-buffer entry (attn_verify_append_q8_host) with
pinned host buffers: each call copies q and the new K/V tokens host->device in one copy,
runs the kernels and reads the output back, eagerly, with no graph.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify-attn us/call and KV-scan GB/s (% HBM peak); prompt-attn TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
VERIFY_T = (4, 8)
HEADLINE_CTX = 20676            # the context the pages' verify speedups are quoted at
EXTRA_CTX = (32768, 4096)       # the largest context, and the 27B-class context with outliers
GRAPH_MAX = 64                  # steps per CUDA graph at most
HEADLINE_WORKLOAD = f"verify-24q4kv-hd256-ctx{HEADLINE_CTX}-T4+T8"
TC_KERNEL_FILES = ["verify_tc.cu", "verify_plan.cuh", "tc.cuh"]   # the code a traffic capture covers


def graph_chunks(n: int, g_max: int = GRAPH_MAX) -> list[tuple[int, int]]:
    """(steps per graph, replays) pairs whose steps add up to exactly n: a graph of
    min(n, g_max) steps replayed n // that many times, plus one graph of the remainder."""
    if n <= 0:
        return []
    g = min(n, g_max)
    out = [(g, n // g)]
    if n % g:
        out.append((n % g, 1))
    return out


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        return summarize_clock_lines(self.lines)


def summarize_clock_lines(lines) -> dict:
    """Median SM clock, maximum SM clock and the throttle reasons seen active, from nvidia-smi
    lines in ClockSampler.FIELDS order (csv, no header, no units); malformed lines are skipped."""
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            smax.append(float(parts[2]))
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower().startswith("active"):
                reasons.add(n)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    from speculative_verify_attention_gb300 import multigpu
    return multigpu.env_world()


def _barrier(world):
    from speculative_verify_attention_gb300 import multigpu
    multigpu.barrier()


def _max_over_ranks(x: float, world: int) -> float:
    from speculative_verify_attention_gb300 import multigpu
    return multigpu.max_over_ranks(x, device="cuda" if world > 1 else None)


def kernel_source_digest(kernel_files) -> str:
    """sha256 of the kernel sources' code with comments, blank lines and spacing removed, so that
    an edit of comments or layout alone keeps a capture valid while any change of code
    invalidates it."""
    import hashlib
    h = hashlib.sha256()
    for name in kernel_files:
        with open(os.path.join(ROOT, "speculative_verify_attention_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(" ".join(line.split()) for line in text.splitlines() if line.strip()).encode())
    return h.hexdigest()


def _kernel_traffic(kernel_files, workload: str):
    """DRAM bytes per launch from the committed ncu capture of `workload`, if the kernel
    code is still the code that capture measured (else None: the counters are stale)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            entry = json.load(f)[workload]
        ok = entry.get("code_sha256") == kernel_source_digest(kernel_files)
        return float(entry["dram_bytes_per_launch"]) if ok else None
    except Exception:
        return None


# ----------------------------------------------------------------------------- oracle arm

def oracle_verify_sample(steps: int, warmup: int, budget_s: float, threads: int | None = None,
                         max_pairs: int = 96):
    """Time the fp64 oracle on (row, q-head) pairs of the headline T=4 verify call (context
    20,676), a bounded sample: one untimed probe batch sets the pairs per step so that `steps`
    steps take about `budget_s` seconds (at least one pair, at most max_pairs).
    Returns (GB/s-equivalent, seconds per step, threads, description)."""
    import oracle
    from speculative_verify_attention_gb300 import workloads

    w = workloads.long_verify(HEADLINE_CTX, 4)
    inp = workloads.make_inputs(w)
    c = oracle.Cache(w.n_kv_heads, w.head_dim, w.kv_len)
    c.append(inp.k, inp.v, 0)
    if threads:
        oracle.set_threads(threads)
    n_thr = oracle.get_threads()
    pairs = [(i, h) for i in range(w.n_q) for h in range(w.n_q_heads)]
    rng = np.random.default_rng(0)

    def run(n):
        sel = [pairs[k] for k in rng.integers(0, len(pairs), n)]
        oracle.attention(c, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, sel=sel)

    t0 = time.perf_counter()
    run(n_thr)                                           # probe: one pair per thread
    per_pair = (time.perf_counter() - t0) / n_thr
    n_pairs = int(max(1, min(max_pairs, budget_s / max(steps, 1) / max(per_pair, 1e-9))))
    for _ in range(warmup):
        run(n_pairs)
    t0 = time.perf_counter()
    for _ in range(steps):
        run(n_pairs)
    dt = time.perf_counter() - t0
    calls = steps * n_pairs / len(pairs)
    gbs = calls * w.kv_bytes() / dt / 1e9
    desc = (f"{n_pairs} random (row, q-head) pairs per step of the {len(pairs)} of the T=4 call at context "
            f"{HEADLINE_CTX} (kv_len {w.kv_len}), {steps} steps; GB/s counts each pair as 1/{len(pairs)} of the "
            f"call's {w.kv_bytes() / 1e6:.2f} MB of K/V")
    return gbs, dt / steps, n_thr, desc


def oracle_sweep() -> None:
    """The fp64 oracle timed per configuration on the host cores (a baseline only): full calls
    of the verify configurations, all OpenMP threads, median of up to three runs, plus a
    one-thread figure scaled from a sample of (row, q-head) pairs; the prompt chunk from a
    sample of pairs at random rows, scaled to the whole chunk.  One JSON line per cell."""
    import oracle
    from speculative_verify_attention_gb300 import workloads

    n_thr = oracle.get_threads()

    def cache_for(w, inp):
        c = oracle.Cache(w.n_kv_heads, w.head_dim, w.kv_len)
        c.append(inp.k, inp.v, 0)
        return c

    def timed(fn, runs):
        ts = []
        for _ in range(runs):
            t0 = time.perf_counter()
            fn()
            ts.append(time.perf_counter() - t0)
        return float(np.median(ts))

    cells = [(workloads.TINY, 3), (workloads.verify_27b(4), 3), (workloads.verify_27b(8), 3),
             (workloads.long_verify(20676, 4), 3), (workloads.long_verify(20676, 8), 1),
             (workloads.long_verify(20676, 32), 1), (workloads.long_verify(32768, 4), 3),
             (workloads.hd128_verify(4), 3)]
    for w, runs in cells:
        inp = workloads.make_inputs(w)
        c = cache_for(w, inp)
        oracle.set_threads(n_thr)
        sec = timed(lambda: oracle.attention(c, inp.q, w.kv_len, w.q_pos0, w.softmax_scale), runs)
        pairs = [(i, h) for i in range(w.n_q) for h in range(w.n_q_heads)]
        sel = [pairs[k] for k in np.random.default_rng(1).integers(0, len(pairs), 4)]
        oracle.set_threads(1)
        sec1 = timed(lambda: oracle.attention(c, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, sel=sel), 1)
        oracle.set_threads(n_thr)
        print(json.dumps({"oracle_cell": w.name, "ms_per_call": sec * 1e3, "runs": runs, "cores": n_thr,
                          "kv_gbs": w.kv_bytes() / sec / 1e9,
                          "ms_per_call_1thread": sec1 * len(pairs) / len(sel) * 1e3,
                          "sample_1thread": f"{len(sel)} of {len(pairs)} pairs, scaled"}), flush=True)
        del c, inp
    for w in (workloads.PROMPT, workloads.PROMPT_HD128):
        inp = workloads.make_inputs(w)
        c = cache_for(w, inp)
        n_pairs = 4 * n_thr
        rng = np.random.default_rng(2)
        sel = [(int(i), int(h)) for i, h in zip(rng.integers(0, w.n_q, n_pairs), rng.integers(0, w.n_q_heads, n_pairs))]
        sec = timed(lambda: oracle.attention(c, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, sel=sel), 1)
        total = w.n_q * w.n_q_heads
        print(json.dumps({"oracle_cell": w.name, "ms_per_call": sec * total / n_pairs * 1e3, "runs": 1,
                          "cores": n_thr, "tflops": w.causal_flops() / (sec * total / n_pairs) / 1e12,
                          "sample": f"{n_pairs} of {total} (query, q-head) pairs at random rows, scaled "
                                    f"to the chunk ({sec:.2f} s timed)"}), flush=True)
        del c, inp


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    gbs, sec, thr, desc = oracle_verify_sample(args.steps, min(args.warmup, 3), budget_s=90.0)
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": HEADLINE_WORKLOAD + " (CPU oracle sample)"},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": thr, "kind": "oracle", "sample": desc},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- native arm

def run_native(args, world, rank, local):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from speculative_verify_attention_gb300 import (PreparedAppendVerifyHost, attn_verify_append_q8,
                                                    attn_verify_append_q8_host_scratch_bytes,
                                                    attn_verify_append_q8_workspace_bytes,
                                                    attn_verify_q8_workspace_bytes, kvq8_device_error, workloads)

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm_peak, bf16_peak, peak_src = _peaks()
    fp16_peak = bf16_peak   # fp16 and bf16 operands share one dense tensor-core rate

    ctx = HEADLINE_CTX
    ws_ = {T: workloads.long_verify(ctx, T) for T in VERIFY_T}
    w0 = ws_[VERIFY_T[0]]
    inp = workloads.make_inputs(ws_[max(VERIFY_T)])     # K/V for ctx + 8 tokens, seeded
    ring = _ring_for(ws_[max(VERIFY_T)], dev, args.ring_l2, inp=inp)
    n_ring = len(ring)
    cache_bytes = _cache_bytes(ring[0])
    q = {T: torch.from_numpy(workloads.make_inputs(ws_[T], kv_len=1).q).to(dev) for T in VERIFY_T}
    knew = {T: torch.from_numpy(inp.k[ctx:ctx + T].copy()).to(dev) for T in VERIFY_T}
    vnew = {T: torch.from_numpy(inp.v[ctx:ctx + T].copy()).to(dev) for T in VERIFY_T}
    del inp
    out = {T: torch.empty_like(q[T]) for T in VERIFY_T}
    wsb = {T: torch.empty(max(attn_verify_q8_workspace_bytes(T, w0.n_q_heads, w0.head_dim, ctx + T, w0.n_kv_heads),
                              attn_verify_append_q8_workspace_bytes(T, w0.n_q_heads, w0.head_dim, ctx,
                                                                    w0.n_kv_heads)),
                          dtype=torch.uint8, device=dev) for T in VERIFY_T}
    kv_bytes_step = sum(ws_[T].kv_bytes() for T in VERIFY_T)

    def step(s):
        # the step's windows are independent problems (their own caches of the ring), run back to
        # back on one stream (measured a little faster than two streams: each call's split kernel
        # fills every SM, and the next call's prologue overlaps the merge kernel before it); each
        # call appends its window's K/V to the cache (fused into the verify kernel) and scans
        # ctx + T keys
        for j, T in enumerate(VERIFY_T):
            c = ring[(s + j * (n_ring // len(VERIFY_T))) % n_ring]
            attn_verify_append_q8(q[T], knew[T], vnew[T], c, ctx, w0.softmax_scale, out=out[T], workspace=wsb[T])

    launches_per_step = len(VERIFY_T) * 2   # verify split (with the append) + combine per T

    timed_chunks = graph_chunks(args.steps)
    warm_chunks = graph_chunks(args.warmup)
    s_ = torch.cuda.Stream(device=dev)
    s_.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s_):
        for i in range(3):
            step(i)
    torch.cuda.current_stream().wait_stream(s_)
    torch.cuda.synchronize()
    graphs = {}
    for g_len, _ in timed_chunks + warm_chunks:
        if g_len not in graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(g_len):
                    step(i)
            graphs[g_len] = g

    def replay(chunks):
        for g_len, reps in chunks:
            for _ in range(reps):
                graphs[g_len].replay()

    replay(warm_chunks)
    torch.cuda.synchronize()
    _barrier(world)
    torch.cuda.synchronize()
    clk = ClockSampler(local)
    clk.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    replay(timed_chunks)
    e1.record()
    torch.cuda.synchronize()
    _barrier(world)
    ms = e0.elapsed_time(e1)

    # per-T cells (one call at a time): the whole call (split + combine) and the split kernel
    # alone, whose time is the roofline's denominator
    per_t = {T: _verify_cell(ws_[T], ring, dev, hbm_peak) for T in VERIFY_T}
    clocks = clk.stop()
    ms = _max_over_ranks(ms, world)
    steps = args.steps
    ms_per_step = ms / steps
    gbs = world * kv_bytes_step * steps / (ms * 1e-3) / 1e9
    del graphs

    # e2e through the C ABI with pinned host buffers, eager: per T one attn_verify_append_q8_host
    # call (q, k_new, v_new copied in with one host-to-device copy, the two kernels, the output
    # copied back)
    h_in = {T: torch.cat([q[T].cpu().reshape(-1), knew[T].cpu().reshape(-1), vnew[T].cpu().reshape(-1)]).pin_memory()
            for T in VERIFY_T}
    h_out = {T: torch.empty(out[T].numel(), dtype=torch.float32).pin_memory() for T in VERIFY_T}
    scratch = {T: torch.empty(attn_verify_append_q8_host_scratch_bytes(T, w0.n_q_heads, w0.head_dim, ctx,
                                                                       w0.n_kv_heads),
                              dtype=torch.uint8, device=dev) for T in VERIFY_T}
    h2d = sum(h_in[T].numel() * 4 for T in VERIFY_T)
    d2h = sum(h_out[T].numel() * 4 for T in VERIFY_T)

    # The two windows of a step are independent problems: each T runs on a stream of its own
    # (so one call's copies overlap the other's kernels) and reads its own cache of the ring.
    # The calls' arguments are marshalled once per (cache, T); a step is one C-ABI call per T.
    e2e_streams = {T: torch.cuda.Stream(device=dev) for T in VERIFY_T}
    prepared = [{T: PreparedAppendVerifyHost(h_in[T], T, w0.n_q_heads, ring[(i + j * n_ring // len(VERIFY_T)) % n_ring],
                                             ctx, w0.softmax_scale, h_out[T], scratch[T], stream=e2e_streams[T])
                 for j, T in enumerate(VERIFY_T)} for i in range(n_ring)]

    def e2e_step(s):
        calls = prepared[s % n_ring]
        for T in VERIFY_T:
            calls[T]()

    e2e_steps = min(steps, 2000)
    for s in range(min(args.warmup, 20)):
        e2e_step(s)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(e2e_steps):
        e2e_step(s)
    torch.cuda.synchronize()
    e2e_sec = _max_over_ranks(time.perf_counter() - t0, world)
    e2e_gbs = world * kv_bytes_step * e2e_steps / e2e_sec / 1e9
    del prepared, ring
    torch.cuda.empty_cache()

    # the other contexts of the family: the largest (32,768) and the 27B-class 4,096 with outliers
    cells = {}
    if not args.no_long_context:
        for c_ in EXTRA_CTX:
            cw = {T: (workloads.long_verify(c_, T) if c_ != 4096 else workloads.verify_27b(T)) for T in VERIFY_T}
            cring = _ring_for(cw[max(VERIFY_T)], dev, args.ring_l2)   # capacity covers every T
            for T in VERIFY_T:
                cells[cw[T].name] = _verify_cell(cw[T], cring, dev, hbm_peak)
            del cring
            torch.cuda.empty_cache()

    # prompt chunk (tensor-core kernel), L2 flushed between timed calls
    prompt = prompt_bench(args, dev, fp16_peak) if not args.no_prompt else None
    if prompt is not None and "unavailable" not in prompt:   # the second prompt shape (hd128, 32q/8kv)
        from speculative_verify_attention_gb300 import workloads as _wl
        torch.cuda.empty_cache()
        prompt["hd128"] = prompt_bench(args, dev, fp16_peak, _wl.PROMPT_HD128)
        torch.cuda.empty_cache()
        prompt["k8v4"] = prompt_bench(args, dev, fp16_peak, _wl.PROMPT, pool="k8v4")
        torch.cuda.empty_cache()
        prompt["f16"] = prompt_bench(args, dev, fp16_peak, _wl.PROMPT, pool="f16")
    head = head_bench(dev, hbm_peak, args.ring_l2) if not args.no_head else None
    quant = quantize_bench(dev, hbm_peak) if not args.no_head else None
    device_error = kvq8_device_error(reset=True)

    result = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cpu_steps = 6
            g_, sec_, thr_, desc_ = oracle_verify_sample(cpu_steps, 1, budget_s=15.0)
            g1, _, _, desc1 = oracle_verify_sample(2, 0, budget_s=4.0, threads=1)   # the one-thread figure
            import oracle
            oracle.set_threads(thr_)
            cpu = {"value": g_, "unit": "GB/s", "cores": thr_, "kind": "oracle", "sample": desc_,
                   "value_1thread": g1, "sample_1thread": desc1 + ", one OpenMP thread"}
        # roofline of the dominant kernel (the split-context verify kernel): the step's K/V bytes
        # over the split kernel's per-launch device time, both T together
        split_us = {T: per_t[T]["split_us_per_launch"] for T in VERIFY_T}
        bytes_per_launch = kv_bytes_step / len(VERIFY_T)
        achieved = kv_bytes_step / (sum(split_us.values()) * 1e-6) / 1e9
        result = {
            "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8 K/V codes (Q8_0); QK fp16 hi+lo on tcgen05, PV fp16 hi+lo on mma.sync, f32 accumulate",
            "data": "synthetic",
            "config": {"workload": HEADLINE_WORKLOAD, "model": None,
                       "global_batch": world, "seq_len": ctx, "verify_rows": list(VERIFY_T),
                       "parallelism": f"replicas x{world}", "l2": f"ring of {n_ring} caches, "
                       f"{n_ring * cache_bytes / 2**20:.0f} MiB > 4x L2 (every step reads a different cache)",
                       "step": "per T in {4,8}: attn_verify_append_q8 (K/V of T new tokens quantised into the "
                               "cache by the verify kernel's window slice; scan over ctx+T); the two windows are "
                               "independent (each on its own cache of the ring), back to back on one stream",
                       "graph": " + ".join(f"{r} x {g}-step graph" for g, r in timed_chunks) + " timed; "
                                + " + ".join(f"{r} x {g}-step graph" for g, r in warm_chunks) + " warm-up"},
            "us_per_call": sum(per_t[T]["us_per_call"] for T in VERIFY_T) / len(VERIFY_T),
            "per_T": {f"T{T}": per_t[T] for T in VERIFY_T},
            "cells": cells,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak,
                         "traffic": _kernel_traffic(TC_KERNEL_FILES, f"verify-24q4kv-hd256-ctx{ctx}-T4+T8"),
                         "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs, burst)",
                         "kernel": "verify_tc_kernel (the split-context verify kernel, timed alone through "
                                   "attn_verify_q8_partials over the same ring)",
                         "algorithmic_bytes_per_launch": bytes_per_launch,
                         "us_per_launch": {f"T{T}": split_us[T] for T in VERIFY_T}},
            "prompt": prompt,
            "verify_head": head,
            "quantize": quant,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_gbs, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "us_per_step": e2e_sec / e2e_steps * 1e6, "steps": e2e_steps,
                    "path": "attn_verify_append_q8_host (C ABI, pinned host buffers, arguments marshalled "
                            "once), eager, one call per T, the two T on two streams"},
            "clocks": clocks,
            "gpu_launches": launches_per_step * steps,
            "device_error_flag": device_error,
        }
    return result


def _cache_bytes(c) -> int:
    return sum(t.numel() * t.element_size() for t in (c.k_codes, c.v_codes, c.k_scales, c.v_scales))


def _verify_cell(w, ring, dev, hbm_peak) -> dict:
    """Per-call device time of attn_verify_q8 on workload w over the ring, and of its split
    kernel alone (attn_verify_q8_partials), each from a CUDA graph of at least 32 calls
    replayed 10 times (median replay)."""
    us = time_verify_cell(w, ring, dev)
    split = time_verify_cell(w, ring, dev, partials=True)
    n_calls = max(len(ring), 32)
    gbs = w.kv_bytes() / (us * 1e-6) / 1e9
    return {"workload": w.name, "us_per_call": us, "kv_gbs": gbs, "hbm_frac": gbs / hbm_peak,
            "split_us_per_launch": split, "split_hbm_frac": w.kv_bytes() / (split * 1e-6) / 1e9 / hbm_peak,
            "kv_bytes": w.kv_bytes(), "calls_timed": 10 * n_calls, "ring": len(ring)}


def head_bench(dev, hbm_peak, ring_l2):
    """argmax_rows_top_prob over T x 248,320 fp32 logits (T = 4, 8, 32): device time per call from
    a CUDA graph walking a ring of logits buffers larger than 4x the L2."""
    import torch

    from speculative_verify_attention_gb300 import argmax_rows_top_prob, load_library
    V = 248320
    res = {}
    for T in (4, 8, 32):
        nbytes = T * V * 4
        n_ring = max(2, int(np.ceil(ring_l2 * L2_BYTES / nbytes)))
        gen = torch.Generator(device=dev).manual_seed(77 + T)
        ring = [torch.randn((T, V), device=dev, generator=gen) * 3.0 for _ in range(n_ring)]
        idx = torch.empty(T, dtype=torch.int32, device=dev)
        top = torch.empty(T, dtype=torch.float32, device=dev)
        ws = torch.empty(max(16, int(load_library().argmax_rows_top_prob_workspace_bytes(T, V))), dtype=torch.uint8,
                         device=dev)
        for i in range(3):
            argmax_rows_top_prob(ring[i % n_ring], workspace=ws, argmax=idx, top_prob=top)
        torch.cuda.synchronize()
        n_calls = max(n_ring, 32)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n_calls):
                argmax_rows_top_prob(ring[i % n_ring], workspace=ws, argmax=idx, top_prob=top)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 10
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / (reps * n_calls)
        gbs = nbytes / (us * 1e-6) / 1e9
        res[f"T{T}"] = {"vocab": V, "us_per_call": us, "logits_gbs": gbs, "hbm_frac": gbs / hbm_peak,
                        "ring": n_ring}
        del ring
        torch.cuda.empty_cache()
    return res


def quantize_bench(dev, hbm_peak):
    """kvq8_append (Q8_0 quantiser, both planes in one launch) of a 32,768-token prefill chunk
    of a 4-KV-head hd256 cache: 67 M values, 268 MB fp32 read and 71 MB written per call, so the
    inputs exceed the L2 and every call streams them from HBM.  Device time per call from CUDA
    events around 20 calls."""
    import torch

    from speculative_verify_attention_gb300 import KVCacheQ8
    n_tok, hkv, hd = 32768, 4, 256
    gen = torch.Generator(device=dev).manual_seed(91)
    k = torch.randn((n_tok, hkv, hd), device=dev, generator=gen)
    v = torch.randn((n_tok, hkv, hd), device=dev, generator=gen)
    cache = KVCacheQ8(hkv, hd, n_tok, device=dev)
    for _ in range(3):
        cache.append(k, v, 0)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 20
    a.record()
    for _ in range(n):
        cache.append(k, v, 0)
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / n
    values = 2 * n_tok * hkv * hd
    nbytes = values * 4 + values + values // 32 * 2
    gbs = nbytes / (us * 1e-6) / 1e9
    del k, v, cache
    torch.cuda.empty_cache()
    return {"workload": f"kvq8_append-{n_tok}tok-{hkv}kv-hd{hd}", "us_per_call": us, "values": values,
            "bytes_per_call": nbytes, "gbs": gbs, "hbm_frac": gbs / hbm_peak,
            "l2": "inputs (268 MB) larger than the L2"}


def prompt_bench(args, dev, fp16_peak, w=None, pool="q8"):
    import torch

    from speculative_verify_attention_gb300 import (KVCacheF16, KVCacheK8V4, KVCacheQ8, KVQ8Error, attn_prompt_f16,
                                                    attn_prompt_f16_workspace_bytes, attn_prompt_k8v4, attn_prompt_q8,
                                                    attn_prompt_q8_workspace_bytes, workloads)
    w = w or workloads.PROMPT
    inp = workloads.make_inputs(w)
    pool_cls = {"q8": KVCacheQ8, "k8v4": KVCacheK8V4, "f16": KVCacheF16}[pool]
    c = pool_cls(w.n_kv_heads, w.head_dim, w.kv_len, device=dev)
    c.append(torch.from_numpy(inp.k).to(dev), torch.from_numpy(inp.v).to(dev), 0)
    attn_prompt_q8 = {"q8": attn_prompt_q8, "k8v4": attn_prompt_k8v4, "f16": attn_prompt_f16}[pool]  # same call shape
    q = torch.from_numpy(inp.q).to(dev)
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    ws_bytes = attn_prompt_q8_workspace_bytes(w.n_q, w.n_q_heads, w.head_dim, w.kv_len, w.q_pos0, w.n_kv_heads)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    # the library's own sizes tell the route: only the two-pass route needs room for an fp16 copy
    two_pass = pool != "f16" and ws_bytes > attn_prompt_f16_workspace_bytes(
        w.n_q, w.n_q_heads, w.head_dim, w.kv_len, w.q_pos0, w.n_kv_heads)
    route = ("fp16 tiles by tensor copy" if pool == "f16" else
             "two-pass: one dequantising pass into an fp16 copy in the workspace, then the tensor-copy kernel"
             if two_pass else "one-pass: tiles dequantised in shared memory")
    try:
        attn_prompt_q8(q, c, w.kv_len, w.q_pos0, w.softmax_scale, out=out, workspace=ws)
    except KVQ8Error as e:
        return {"unavailable": str(e)}
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    times = []
    n = max(3, min(args.prompt_steps, 20))
    for i in range(n + 2):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        attn_prompt_q8(q, c, w.kv_len, w.q_pos0, w.softmax_scale, out=out, workspace=ws)
        b.record()
        torch.cuda.synchronize()
        if i >= 2:
            times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    tf = w.causal_flops() / (ms * 1e-3) / 1e12
    return {"workload": w.name, "pool": pool, "ms_per_call": ms, "tflops": tf, "peak_tflops": fp16_peak,
            "frac": tf / fp16_peak, "peak_source": "MEASURED_PEAKS.json bf16_tflops (cuBLAS bf16, burst); fp16 "
            "and bf16 share one dense tensor-core rate", "dtype": "fp16 operands, single pass (q, K, P, V "
            "each one fp16 value, not split hi+lo), f32 accumulate",
            "flops": w.causal_flops(), "calls_timed": n, "l2": "flushed (256 MiB write) before every call",
            "route": route, "workspace_bytes": ws_bytes}


def _ring_for(w, dev, ring_l2, inp=None):
    import torch

    from speculative_verify_attention_gb300 import KVCacheQ8, workloads
    inp = inp if inp is not None else workloads.make_inputs(w)
    base = KVCacheQ8(w.n_kv_heads, w.head_dim, w.kv_len, device=dev)
    base.append(torch.from_numpy(inp.k).to(dev), torch.from_numpy(inp.v).to(dev), 0)
    nbytes = sum(t.numel() * t.element_size() for t in (base.k_codes, base.v_codes, base.k_scales, base.v_scales))
    n_ring = max(2, int(np.ceil(ring_l2 * L2_BYTES / nbytes)))
    ring = [base]
    for _ in range(n_ring - 1):
        c = KVCacheQ8(w.n_kv_heads, w.head_dim, w.kv_len, device=dev)
        for a, b in ((c.k_codes, base.k_codes), (c.v_codes, base.v_codes), (c.k_scales, base.k_scales),
                     (c.v_scales, base.v_scales)):
            a.copy_(b)
        ring.append(c)
    return ring


def _ring_f16(w, dev, ring_l2):
    """A ring of fp16 pools holding the workload's K/V (total size above ring_l2 x L2)."""
    import torch

    from speculative_verify_attention_gb300 import KVCacheF16, workloads
    inp = workloads.make_inputs(w)
    base = KVCacheF16(w.n_kv_heads, w.head_dim, w.kv_len, device=dev)
    base.append(torch.from_numpy(inp.k).to(dev), torch.from_numpy(inp.v).to(dev), 0)
    nbytes = 2 * base.k.numel() * base.k.element_size()
    ring = [base]
    for _ in range(max(2, int(np.ceil(ring_l2 * L2_BYTES / nbytes))) - 1):
        c = KVCacheF16(w.n_kv_heads, w.head_dim, w.kv_len, device=dev)
        c.k.copy_(base.k)
        c.v.copy_(base.v)
        ring.append(c)
    return ring


def _ring_k8v4(w, dev, ring_l2):
    """A ring of K8V4 pools holding the workload's K/V (total size above ring_l2 x L2)."""
    import torch

    from speculative_verify_attention_gb300 import KVCacheK8V4, workloads
    inp = workloads.make_inputs(w)
    base = KVCacheK8V4(w.n_kv_heads, w.head_dim, w.kv_len, device=dev)
    base.append(torch.from_numpy(inp.k).to(dev), torch.from_numpy(inp.v).to(dev), 0)
    planes = ("k_codes", "k_scales", "v_codes", "v_scales")
    nbytes = sum(getattr(base, n).numel() * getattr(base, n).element_size() for n in planes)
    ring = [base]
    for _ in range(max(2, int(np.ceil(ring_l2 * L2_BYTES / nbytes))) - 1):
        c = KVCacheK8V4(w.n_kv_heads, w.head_dim, w.kv_len, device=dev)
        for n in planes:
            getattr(c, n).copy_(getattr(base, n))
        ring.append(c)
    return ring


def k8v4_kv_bytes(w) -> int:
    """Bytes of the K8V4 planes read for kv_len tokens: Q8_0 K, 4-bit V, fp16 scales for both."""
    hd = w.head_dim
    return w.n_kv_heads * w.kv_len * (hd + hd // 16 + hd // 2 + hd // 16)


def f16_kv_bytes(w) -> int:
    """Bytes of the fp16 K and V planes read for kv_len tokens."""
    return 2 * w.n_kv_heads * w.kv_len * w.head_dim * 2


def binary_tree_mask(T: int) -> np.ndarray:
    """Window mask of a binary draft tree of T tokens (node i's parent is (i - 1) // 2): each row
    sees its ancestors and itself."""
    masks = []
    for i in range(T):
        m, a = 0, i
        while a >= 0:
            m |= 1 << a
            a = (a - 1) // 2 if a > 0 else -1
        masks.append(m)
    return np.array(masks, dtype=np.uint32)


def time_verify_cell(w, ring, dev, reps=10, tree_mask=None, partials=False):
    """Device time per attn_verify_q8 call (attn_verify_tree_q8 when a window mask is given;
    attn_verify_q8_partials, the split kernel alone, with partials=True):
    a CUDA graph of at least 32 calls walking the ring (total size > 4x L2, so K/V come from
    HBM; a one-cache ring gives the warm-L2 time) is replayed `reps` times, each replay timed
    with CUDA events; returns the median over the replays of microseconds per call."""
    import torch

    from speculative_verify_attention_gb300 import (KVCacheF16, KVCacheK8V4, attn_verify_f16, attn_verify_k8v4,
                                                    attn_verify_q8, attn_verify_q8_partials,
                                                    attn_verify_q8_partials_count, attn_verify_q8_workspace_bytes,
                                                    attn_verify_tree_q8, workloads)
    q = torch.from_numpy(workloads.make_inputs(w, kv_len=1).q).to(dev)
    out = torch.empty_like(q)
    ws = torch.empty(attn_verify_q8_workspace_bytes(w.n_q, w.n_q_heads, w.head_dim, w.kv_len, w.n_kv_heads),
                     dtype=torch.uint8, device=dev)
    if isinstance(ring[0], KVCacheF16):   # fp16 pools (the same workspace size rule)
        def call(c):
            attn_verify_f16(q, c, w.kv_len, w.q_pos0, w.softmax_scale, out=out, workspace=ws)
    elif isinstance(ring[0], KVCacheK8V4):
        def call(c):
            attn_verify_k8v4(q, c, w.kv_len, w.q_pos0, w.softmax_scale, out=out, workspace=ws)
    elif partials:
        n = attn_verify_q8_partials_count(w.n_q, w.n_q_heads, w.head_dim, w.kv_len, w.n_kv_heads)
        po = torch.empty((n, w.n_q * w.n_q_heads, w.head_dim), dtype=torch.float32, device=dev)
        pml = torch.empty((n, w.n_q * w.n_q_heads, 2), dtype=torch.float32, device=dev)

        def call(c):
            attn_verify_q8_partials(q, c, w.kv_len, w.q_pos0, w.softmax_scale, part_o=po, part_ml=pml)
    elif tree_mask is not None:
        m = torch.from_numpy(np.ascontiguousarray(tree_mask, np.uint32).view(np.int32)).to(dev)

        def call(c):
            attn_verify_tree_q8(q, c, w.kv_len, w.q_pos0, m, w.softmax_scale, out=out, workspace=ws)
    else:
        def call(c):
            attn_verify_q8(q, c, w.kv_len, w.q_pos0, w.softmax_scale, out=out, workspace=ws)
    for i in range(3):
        call(ring[i % len(ring)])
    torch.cuda.synchronize()
    n_calls = max(len(ring), 32)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n_calls):
            call(ring[i % len(ring)])
    g.replay()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record()
    for r in range(reps):
        g.replay()
        ev[r + 1].record()
    torch.cuda.synchronize()
    per = sorted(ev[r].elapsed_time(ev[r + 1]) * 1e3 / n_calls for r in range(reps))
    return per[reps // 2]


def sweep(args):
    """Verify latency and KV-scan bandwidth per (context, T) cell of the long-context and
    hd128 workload families (one JSON line per cell; not the headline line)."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from speculative_verify_attention_gb300 import workloads
    hbm_peak, bf16_peak, _ = _peaks()
    dev = torch.device("cuda", 0)
    cells = [workloads.verify_27b(t) for t in workloads.VERIFY_27B_T]
    cells += [workloads.long_verify(c, t) for c in workloads.LONG_CTX for t in workloads.LONG_T]
    cells += [workloads.hd128_verify(t) for t in workloads.HD128_T]
    # tree-shaped windows (binary draft trees) on the 27B-class shape
    cells += [(workloads.verify_27b(t), "tree-binary") for t in (8, 16)]
    # fp16 KV pools
    cells += [(workloads.verify_27b(t), "f16") for t in (4, 8)]
    cells += [(workloads.long_verify(c, t), "f16") for c in (20676, 32768) for t in (4, 8)]
    cells += [(workloads.hd128_verify(t), "f16") for t in (4, 8)]
    # K8V4 pools
    cells += [(workloads.verify_27b(t), "k8v4") for t in (4, 8)]
    cells += [(workloads.long_verify(c, t), "k8v4") for c in (20676, 32768) for t in (4, 8)]
    cells += [(workloads.hd128_verify(t), "k8v4") for t in (4, 8)]
    cells = [c if isinstance(c, tuple) else (c, None) for c in cells]
    cells = [(w, kind) for w, kind in cells
             if not args.sweep_filter or re.search(args.sweep_filter, f"{kind}-{w.name}" if kind else w.name)]
    key, ring = None, None
    for w, kind in cells:
        pool = kind if kind in ("f16", "k8v4") else "q8"
        if key != (pool, w.n_kv_heads, w.head_dim, w.kv_len):
            ring = None
            torch.cuda.empty_cache()
            ring = {"f16": _ring_f16, "k8v4": _ring_k8v4, "q8": _ring_for}[pool](w, dev, args.ring_l2)
            key = (pool, w.n_kv_heads, w.head_dim, w.kv_len)
        mask = binary_tree_mask(w.n_q) if kind == "tree-binary" else None
        us = time_verify_cell(w, ring, dev, tree_mask=mask)
        us_warm = time_verify_cell(w, ring[:1], dev, tree_mask=mask)
        kv_bytes = {"f16": f16_kv_bytes, "k8v4": k8v4_kv_bytes, "q8": lambda w_: w_.kv_bytes()}[pool](w)
        gbs = kv_bytes / (us * 1e-6) / 1e9
        # roofline of the cell: K/V bytes at the HBM peak, or the causal flops doubled by the
        # fp16 hi + lo split at the dense tensor peak, whichever takes longer
        t_hbm = kv_bytes / (hbm_peak * 1e9)
        t_tensor = 2 * w.causal_flops() / (bf16_peak * 1e12)
        print(json.dumps({"workload": f"{kind}-{w.name}" if kind else w.name, "us_per_call": us,
                          "kv_mb": kv_bytes / 1e6, "kv_gbs": gbs, "hbm_frac": gbs / hbm_peak,
                          "tflops_alg": w.causal_flops() / (us * 1e-6) / 1e12,
                          "roofline_bound": "hbm" if t_hbm >= t_tensor else "tensor",
                          "roofline_frac": max(t_hbm, t_tensor) / (us * 1e-6),
                          "us_per_call_warm_l2": us_warm, "ring": len(ring)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2048)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--ring-l2", type=float, default=4.2, help="ring size in multiples of the L2")
    ap.add_argument("--prompt-steps", type=int, default=20)
    ap.add_argument("--no-prompt", action="store_true")
    ap.add_argument("--no-head", action="store_true", help="skip the verify-head (argmax / top probability) timing")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-long-context", action="store_true")
    ap.add_argument("--sweep", action="store_true", help="per-cell verify sweep instead of the headline line")
    ap.add_argument("--prompt-only", action="store_true", help="time only the prompt-chunk kernel")
    ap.add_argument("--oracle-sweep", action="store_true",
                    help="time the fp64 CPU oracle per configuration (host cores only, no GPU)")
    ap.add_argument("--sweep-filter", default="", help="with --sweep: time only the cells whose name matches "
                    "this regular expression")
    ap.add_argument("--prompt-filter", default="", help="with --prompt-only: time only the cells whose "
                    "'<pool>-<workload>' name contains this")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = _dist()
    if args.oracle_sweep:
        oracle_sweep()
        return 0
    if args.sweep:
        sweep(args)
        return 0
    if args.prompt_only:
        import torch

        import __graft_entry__
        __graft_entry__.build()
        hbm_peak, bf16_peak, _ = _peaks()
        from speculative_verify_attention_gb300 import workloads as _wl
        for w, pool in ((_wl.PROMPT, "q8"), (_wl.PROMPT_HD128, "q8"), (_wl.PROMPT, "k8v4"), (_wl.PROMPT, "f16"),
                        (_wl.PROMPT_HD128, "f16"), (_wl.PROMPT_HD128, "k8v4")):
            if args.prompt_filter and args.prompt_filter not in f"{pool}-{w.name}":
                continue
            print(json.dumps(prompt_bench(args, torch.device("cuda", 0), bf16_peak, w, pool)), flush=True)
        return 0
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    res = run_native(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
