#!/usr/bin/env python3
"""Benchmark of the hot path on B300: split-KV decode at S = 131072 and the
fused causal prefill at S = 16384.

One step = one pass of the path over one batch of synthetic input:
  1. one decode token (ta_decode_ex): the KV-chunk plan, the split-KV
     partials of every (KV head, chunk) and their log-sum-exp merge -- one
     launch, since the decode kernel merges up to 128 chunks itself;
  2. the causal prefill of the prefill workload (ta_prefill_causal).
Each phase is a CUDA graph replay bracketed by CUDA events on the stream it
is launched on.

The JSON line's ``value`` is decode KV-cache throughput in GB/s (the K and V
bytes a decode step must read, over the time of step 1), summed over ranks;
``us_per_token`` is the decode time of one step; ``prefill_tflops`` the
causal FLOPs over the prefill time.  Inputs are larger than L2 (512 MiB of
K/V per decode step), so no flush is needed between steps.

``--impl reference`` times the float64 CPU oracle on the host cores on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# The headline metric, printed identically by both arms so the two lines compare.
METRIC = "decode KV-cache GB/s (% of B300 HBM peak) and \u00b5s/token at S=128K; prefill TFLOP/s"
DECODE_WORKLOAD = "gqa_32x8_d128_s131072"
WORKLOAD_DESC = (f"{DECODE_WORKLOAD}: B=1, Hq=32, Hkv=8, D=128, S=131072, bf16 q/K/V N(0,1), "
                 f"scale=1/sqrt(128)")
PREFILL_WORKLOAD = "causal_prefill_32x8_d128_s16384"
PROFILES = {  # committed ncu summaries: (file, kernel sources they were taken on)
    "decode": ("decode_tc_kernel_gqa_32x8_d128_s131072.md",
               ("decode_tc.cu", "decode_tc_common.cuh", "common.cuh", "tcgen05.cuh")),
    "prefill": ("prefill_causal_kernel_causal_prefill_32x8_d128_s16384.md",
                ("prefill.cu", "common.cuh", "tcgen05.cuh")),
}


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", device_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        rows = [l for (t, l) in self.lines if t0 - 0.05 <= t <= t1 + 0.05] or [l for (_, l) in self.lines]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def profiled_traffic(which):
    """DRAM bytes per launch of a kernel from its committed ncu summary, if the
    kernel source is unchanged since that capture; else None."""
    name, src_names = PROFILES[which]
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
    except OSError:
        return None
    kv = {}
    for line in text.splitlines():
        if ":" in line and line.startswith("- "):
            key, _, val = line[2:].partition(":")
            kv[key.strip()] = val.strip().strip("`")
    for src_name in src_names:
        src = os.path.join(ROOT, "long_context_decode_04_b300", "csrc", src_name)
        if kv.get(f"{src_name} sha256") != source_hash(src):
            return None
    try:
        return int(kv["dram bytes per launch"])
    except (KeyError, ValueError):
        return None


def reduce_max(val, world, device):
    """The largest of the ranks' values (every rank gets it); the job's time is
    its slowest replica's."""
    if world == 1:
        return val
    import torch
    import torch.distributed as dist
    t = torch.tensor([val], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank, world, seconds_max):
    """Whole-job throughput of `world` independent replicas (weak scaling):
    every rank processes units_per_rank in at most seconds_max."""
    return world * units_per_rank / seconds_max


def measure_varlen(ta, synth, accounting, peaks, dev, reps=20):
    """Decode of the 16-sequence variable-length workload (lengths 1K-32K),
    with a contiguous and a paged (64-key pages) KV cache: median of `reps`
    graph replays each, KV bytes of the attended keys only."""
    import torch
    w = synth.WORKLOADS["varlen_b16_32x8_d128_s1k_32k"]
    x = synth.make_inputs(w)
    lens = [int(v) for v in x["seqlens"]]
    kv_bytes = accounting.decode_kv_bytes(w.B, w.Hkv, w.D, lens, 2)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    sl = x["seqlens"].to(dev)
    kp, vp, bt = synth.to_pages(x["k"], x["v"], lens, 64, seed=11)
    kp, vp, bt = kp.to(dev), vp.to(dev), bt.to(dev)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    ws = ta.decode_workspace(w.B, w.Hq, w.Hkv, w.S, w.D, varlen=True, device=dev)
    calls = {
        "contiguous": lambda: ta.decode(q, k, v, seqlens=sl, scale=w.scale, workspace=ws, out=out, lse=lse),
        "paged_64": lambda: ta.decode_paged(q, kp, vp, bt, sl, scale=w.scale, workspace=ws, out=out, lse=lse),
    }
    res = {"workload": "B=16, Hq=32, Hkv=8, D=128, lengths uniform in [1024, 32768] (seeded), bf16",
           "attended_kv_bytes": kv_bytes}
    stream = torch.cuda.current_stream(dev)
    for name, fn in calls.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        us = sorted(1e3 * a.elapsed_time(b) for a, b in ev)[reps // 2]
        gbs = kv_bytes / (us / 1e6) / 1e9
        res[name] = {"us": round(us, 2), "gbs": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4)}
    return res


def measure_pi(ta, accounting, peaks, dev, w, q, k, v, window=4096, period=64, reps=20):
    """Decode of the 128K-token workload over the pi-Attention key set (the last
    `window` keys plus every `period`-th key before them): median of `reps`
    graph replays, KV bytes of the attended keys only."""
    import torch
    i = w.S - 1
    w0 = max(0, i - window)
    n_keys = (i - w0 + 1) + sum(1 for j in range(i - period, -1, -period) if j < w0)
    kv_bytes = accounting.decode_kv_bytes(w.B, w.Hkv, w.D, n_keys, 2)
    ws = ta.decode_pi_workspace(w.B, w.Hq, w.Hkv, w.S, w.D, window, period, device=dev)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    fn = lambda: ta.decode_pi(q, k, v, window, period, scale=w.scale, workspace=ws, out=out, lse=lse)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    stream = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    us = sorted(1e3 * a.elapsed_time(b) for a, b in ev)[reps // 2]
    gbs = kv_bytes / (us / 1e6) / 1e9
    return {"workload": f"B=1, Hq=32, Hkv=8, D=128, S={w.S}, window={window}, period={period}",
            "attended_keys": n_keys, "attended_kv_bytes": kv_bytes, "us": round(us, 2), "gbs": round(gbs, 1),
            "frac": round(gbs / peaks["hbm_gbs"], 4)}


def measure_other_configs(ta, synth, accounting, peaks, dev, reps=7, inner=10):
    """Decode of the single-head fp32 workload (4096 keys, D = 64) and of the
    1M-key GQA workload with its forced 256-key chunks (4096 splits, merged in
    two levels by the merge kernel): the median over `reps` groups of the mean
    of `inner` back-to-back graph replays (a group between two events, so the
    events' resolution does not bound a short launch), all KV bytes; the
    first-level partials (m, l, o written by the split phase and read back by
    the merge) are reported beside them."""
    import torch
    res = {}
    for name in ("single_head_d64_s4096_f32", "gqa_32x8_d128_s1048576_c256"):
        w = synth.WORKLOADS[name]
        x = synth.make_inputs(w)
        q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
        del x
        chunk = w.chunk or 0
        plan = ta.plan_decode(w.B, w.Hq, w.Hkv, w.S, w.D, chunk=chunk)
        kv_bytes = accounting.decode_kv_bytes(w.B, w.Hkv, w.D, w.S, 4 if w.dtype == "f32" else 2)
        ws = ta.decode_workspace(w.B, w.Hq, w.Hkv, w.S, w.D, chunk=chunk, device=dev)
        out = torch.empty((w.B, w.Hq, w.D), dtype=q.dtype, device=dev)
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)

        def fn():
            ta.decode(q, k, v, scale=w.scale, chunk=chunk, workspace=ws, out=out, lse=lse)

        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        stream = torch.cuda.current_stream(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            a.record(stream)
            for _ in range(inner):
                g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        us = sorted(1e3 * a.elapsed_time(b) / inner for a, b in ev)[reps // 2]
        gbs = kv_bytes / (us / 1e6) / 1e9
        pbytes = accounting.partial_bytes(w.B, w.Hq, plan.n_split, w.D) if plan.n_split > 1 else 0
        res[name] = {"workload": f"B={w.B}, Hq={w.Hq}, Hkv={w.Hkv}, D={w.D}, S={w.S}, {w.dtype}",
                     "n_split": plan.n_split, "chunk": plan.chunk,
                     "launches": 1 + plan.levels,
                     "kv_bytes": kv_bytes, "us": round(us, 2), "gbs": round(gbs, 1),
                     "frac": round(gbs / peaks["hbm_gbs"], 4),
                     "partial_bytes": pbytes,
                     "frac_with_partials": round((kv_bytes + pbytes) / (us / 1e6) / 1e9 / peaks["hbm_gbs"], 4)}
        del q, k, v, ws, out, lse, g
        torch.cuda.empty_cache()
    return res


def measure_fp8(ta, synth, accounting, peaks, dev, w, x, reps=20):
    """Decode of the 128K-token workload with its K/V quantised to E4M3 (one
    factor per KV head): median of `reps` graph replays, KV bytes read (1 byte
    an element)."""
    import torch
    k8, ks = synth.to_e4m3(x["k"])
    v8, vs = synth.to_e4m3(x["v"])
    q = x["q"].to(dev)
    k8, v8, ks, vs = k8.to(dev), v8.to(dev), ks.to(dev), vs.to(dev)
    kv_bytes = accounting.decode_kv_bytes(w.B, w.Hkv, w.D, w.S, 1)
    ws = ta.decode_workspace(w.B, w.Hq, w.Hkv, w.S, w.D, device=dev)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    fn = lambda: ta.decode_fp8(q, k8, v8, k_scale=ks, v_scale=vs, scale=w.scale, workspace=ws, out=out, lse=lse)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    stream = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    us = sorted(1e3 * a.elapsed_time(b) for a, b in ev)[reps // 2]
    gbs = kv_bytes / (us / 1e6) / 1e9
    return {"workload": "B=1, Hq=32, Hkv=8, D=128, S=131072, K/V E4M3 with per-KV-head factors, bf16 q",
            "kv_bytes": kv_bytes, "us": round(us, 2), "gbs": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4)}


def measure_nvfp4(ta, synth, accounting, peaks, dev, w, x, reps=20):
    """Decode of the 128K-token workload with its K/V quantised to NVFP4 (E2M1
    codes, one E4M3 scale per 16 elements, one factor per KV head): median of
    `reps` graph replays; bytes read: 0.5 per element plus 1/16 for the block
    scales."""
    import torch
    k4, kbs, kf = synth.to_nvfp4(x["k"])
    v4, vbs, vf = synth.to_nvfp4(x["v"])
    q = x["q"].to(dev)
    k4, kbs, kf, v4, vbs, vf = (t.to(dev) for t in (k4, kbs, kf, v4, vbs, vf))
    kv_bytes = 2 * w.B * w.Hkv * w.S * (w.D // 2 + w.D // 16)
    ws = ta.decode_workspace(w.B, w.Hq, w.Hkv, w.S, w.D, device=dev)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    fn = lambda: ta.decode_nvfp4(q, k4, v4, kbs, vbs, k_factor=kf, v_factor=vf, scale=w.scale, workspace=ws,
                                 out=out, lse=lse)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    stream = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    us = sorted(1e3 * a.elapsed_time(b) for a, b in ev)[reps // 2]
    gbs = kv_bytes / (us / 1e6) / 1e9
    return {"workload": "B=1, Hq=32, Hkv=8, D=128, S=131072, K/V NVFP4 (E2M1 + E4M3 per 16 elements + fp32 per KV "
                        "head), bf16 q",
            "kv_bytes": kv_bytes, "us": round(us, 2), "gbs": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4)}


def measure_prefill_varlen(ta, synth, peaks, dev, reps=5):
    """Causal prefill of 8 packed sequences with lengths uniform in [1024, 16384]
    (seeded), 32 heads / 8 KV heads: median of `reps` graph replays."""
    import numpy as np
    import torch
    rng = np.random.Generator(np.random.PCG64(1005))
    lens = [int(x) for x in rng.integers(1024, 16384, size=8, endpoint=True)]
    T, H, Hkv, D = sum(lens), 32, 8, 128
    w = synth.Workload("packed_prefill", 5, "prefill", 1, H, Hkv, T, D, "bf16")
    x = synth.make_inputs(w)
    q = x["q"][0].transpose(0, 1).contiguous().to(dev)
    k = x["k"][0].transpose(0, 1).contiguous().to(dev)
    v = x["v"][0].transpose(0, 1).contiguous().to(dev)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    flops = sum(4 * D * H * (L * (L + 1) // 2) for L in lens)
    fn = lambda: ta.prefill_causal_varlen(q, k, v, cu, max(lens), scale=w.scale, out=out, lse=lse)
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    stream = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    ms = sorted(a.elapsed_time(b) for a, b in ev)[reps // 2]
    tf = flops / (ms / 1e3) / 1e12
    return {"workload": f"8 packed sequences, lengths {lens}, H=32, Hkv=8, D=128, causal, bf16",
            "flops": flops, "ms": round(ms, 3), "tflops": round(tf, 1),
            "frac": round(tf / peaks["bf16_tflops"], 4),
            "frac_sustained": round(tf / peaks["bf16_tflops_sustained"], 4)}


def cpu_oracle_decode(x, rows, threads):
    import oracle
    t = time.perf_counter()
    oracle.decode(x["q"], x["k"], x["v"], x["scale"], rows=rows, threads=threads)
    return time.perf_counter() - t


def cpu_baseline_figures(synth, accounting, x2, reps=3):
    """The oracle as it stands on the host cores: one warm-up call, then the
    median of `reps` calls of one full decode step of the 128K workload with all
    the threads the oracle uses (one per query head, up to the core count), and
    single-thread times of one full decode step of the 128K workload and of the
    single-head D = 64 workload (one call each after a warm-up)."""
    import oracle
    w2 = synth.WORKLOADS[DECODE_WORKLOAD]
    rows2 = list(range(w2.Hq))
    threads = min(oracle.default_threads(), len(rows2))
    bytes2 = accounting.decode_kv_bytes(w2.B, w2.Hkv, w2.D, w2.S, 2)
    cpu_oracle_decode(x2, rows2, threads)
    t_mt = statistics.median(cpu_oracle_decode(x2, rows2, threads) for _ in range(reps))
    w1 = synth.WORKLOADS["single_head_d64_s4096_f32"]
    x1 = synth.make_inputs(w1)
    bytes1 = accounting.decode_kv_bytes(w1.B, w1.Hkv, w1.D, w1.S, 4)
    cpu_oracle_decode(x1, [0], 1)
    t1 = statistics.median(cpu_oracle_decode(x1, [0], 1) for _ in range(5))
    t2 = cpu_oracle_decode(x2, rows2, 1)
    return {
        "value": round(bytes2 / t_mt / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
        "sample": f"one full decode step of {DECODE_WORKLOAD} (all 32 query heads over all 131072 keys, "
                  f"512 MiB of K/V): median of {reps} calls after one warm-up, {threads} threads",
        "ms_per_step": round(1e3 * t_mt, 2),
        "single_thread": {
            DECODE_WORKLOAD: {"ms_per_step": round(1e3 * t2, 1), "gbs": round(bytes2 / t2 / 1e9, 4)},
            "single_head_d64_s4096_f32": {"ms_per_step": round(1e3 * t1, 3), "gbs": round(bytes1 / t1 / 1e9, 4)},
        },
    }


def run_reference(args, rank, world):
    """The float64 CPU oracle on the host cores, a bounded sample per step."""
    if rank != 0:
        return
    import oracle
    from long_context_decode_04_b300 import accounting, synth
    w = synth.WORKLOADS[DECODE_WORKLOAD]
    x = synth.make_inputs(w)
    rows = list(range(w.Hq))  # a whole decode step: every query head over every key
    threads = min(oracle.default_threads(), len(rows))
    sample_bytes = accounting.decode_kv_bytes(w.B, w.Hkv, w.D, w.S, 2)
    for _ in range(args.warmup):
        cpu_oracle_decode(x, rows, threads)
    t = 0.0
    for _ in range(args.steps):
        t += cpu_oracle_decode(x, rows, threads)
    gbs = sample_bytes * args.steps / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4),
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t / args.steps, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": "per step: one full decode step, all 32 query heads over all "
                                       "131072 keys (512 MiB of K/V); the oracle threads over query heads"},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_launches(which, n):
    """A few plain launches of one workload and nothing else (no timing, no
    JSON): the command the ncu captures in profiles/ run.  `which` is one of
    decode (the 128K-token GQA decode), fp8 (the same over an E4M3 cache),
    nvfp4 (the same over an NVFP4 cache),
    paged (the 16-sequence variable-length decode in 64-key pages), prefill
    (the 16K-token causal prefill)."""
    import torch
    from long_context_decode_04_b300 import synth, ta
    dev = torch.device("cuda", 0)
    if which == "prefill":
        pw = synth.WORKLOADS[PREFILL_WORKLOAD]
        y = synth.make_inputs(pw)
        pq, pk, pv = (y[n].to(dev) for n in ("q", "k", "v"))
        fn = lambda: ta.prefill_causal(pq, pk, pv, scale=pw.scale)
    elif which == "paged":
        w = synth.WORKLOADS["varlen_b16_32x8_d128_s1k_32k"]
        x = synth.make_inputs(w)
        lens = [int(v) for v in x["seqlens"]]
        kp, vp, bt = synth.to_pages(x["k"], x["v"], lens, 64, seed=11)
        q, kp, vp, bt = x["q"].to(dev), kp.to(dev), vp.to(dev), bt.to(dev)
        sl = x["seqlens"].to(dev)
        fn = lambda: ta.decode_paged(q, kp, vp, bt, sl, scale=w.scale)
    else:
        w = synth.WORKLOADS[DECODE_WORKLOAD]
        x = synth.make_inputs(w)
        q = x["q"].to(dev)
        if which == "fp8":
            k8, ks = synth.to_e4m3(x["k"])
            v8, vs = synth.to_e4m3(x["v"])
            k8, ks, v8, vs = k8.to(dev), ks.to(dev), v8.to(dev), vs.to(dev)
            fn = lambda: ta.decode_fp8(q, k8, v8, k_scale=ks, v_scale=vs, scale=w.scale)
        elif which == "nvfp4":
            k4, kbs, kf = (t.to(dev) for t in synth.to_nvfp4(x["k"]))
            v4, vbs, vf = (t.to(dev) for t in synth.to_nvfp4(x["v"]))
            fn = lambda: ta.decode_nvfp4(q, k4, v4, kbs, vbs, k_factor=kf, v_factor=vf, scale=w.scale)
        else:
            k, v = x["k"].to(dev), x["v"].to(dev)
            fn = lambda: ta.decode(q, k, v, scale=w.scale)
    for _ in range(n):
        fn()
    torch.cuda.synchronize()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-prefill", action="store_true", help="time the decode path only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-extra", action="store_true", help="skip the variable-length / paged decode figures")
    ap.add_argument("--launches", choices=["decode", "fp8", "nvfp4", "paged", "prefill"],
                    help="only make --steps plain launches of one workload (for profilers); prints nothing")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    rank, world, local = dist_env()

    if args.launches:
        run_launches(args.launches, args.steps)
        return

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import torch.distributed as dist

    from long_context_decode_04_b300 import accounting, synth, ta

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    peaks = load_peaks()
    stream = torch.cuda.current_stream(dev)

    # ---------------- decode workload (each rank runs an independent replica)
    w = synth.WORKLOADS[DECODE_WORKLOAD]
    x = synth.make_inputs(w)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    plan = ta.plan_decode(w.B, w.Hq, w.Hkv, w.S, w.D)
    ws = ta.decode_workspace(w.B, w.Hq, w.Hkv, w.S, w.D, device=dev)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    kv_bytes = accounting.decode_kv_bytes(w.B, w.Hkv, w.D, w.S, 2)
    # up to 128 chunks the decode kernel merges them itself: one launch
    decode_launches = 1 + plan.levels

    # ---------------- prefill workload
    do_prefill = not args.no_prefill
    pf = None
    if do_prefill:
        pw = synth.WORKLOADS[PREFILL_WORKLOAD]
        y = synth.make_inputs(pw)
        pq, pk, pv = (y[n].to(dev) for n in ("q", "k", "v"))
        pout = torch.empty_like(pq)
        plse = torch.empty((pw.B, pw.Hq, pw.S), dtype=torch.float32, device=dev)
        try:
            ta.prefill_causal(pq, pk, pv, scale=pw.scale, out=pout, lse=plse)
            torch.cuda.synchronize()
            pf = (pw, pq, pk, pv, pout, plse)
        except ta.TAError as e:
            if e.status != ta.TA_ERR_UNSUPPORTED:
                raise
            do_prefill = False
    launches_per_step = decode_launches + (1 if do_prefill else 0)

    def run_decode():
        ta.decode(q, k, v, scale=w.scale, workspace=ws, out=out, lse=lse)

    def run_prefill():
        pw_, pq_, pk_, pv_, pout_, plse_ = pf
        ta.prefill_causal(pq_, pk_, pv_, scale=pw_.scale, out=pout_, lse=plse_)

    for _ in range(args.warmup):
        run_decode()
        if do_prefill:
            run_prefill()
    torch.cuda.synchronize()

    # Each phase is captured once into a CUDA graph, so that a timed step is
    # a couple of graph launches and the host never holds the GPU back: the
    # events between replays then measure device time only.
    graphs = []
    for fn in (run_decode,) + ((run_prefill,) if do_prefill else ()):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs.append(g)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)

    def step(ev):
        ev[0].record(stream)
        graphs[0].replay()
        ev[1].record(stream)
        if do_prefill:
            graphs[1].replay()
        ev[2].record(stream)

    def new_events():
        return [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    warm = new_events()
    for _ in range(args.warmup):
        step(warm)
    torch.cuda.synchronize()

    props = torch.cuda.get_device_properties(dev)
    dev_id = str(getattr(props, "uuid", "")) or str(local)
    if dev_id and not dev_id.startswith("GPU-") and len(dev_id) == 36:
        dev_id = "GPU-" + dev_id
    sampler = ClockSampler(dev_id)
    time.sleep(0.3)  # let the sampler start before the timed region

    evs = [new_events() for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    wall1 = time.time()
    clocks = sampler.stop(wall0, wall1)

    total_ms = t_start.elapsed_time(t_end)
    dec_ms = [e[0].elapsed_time(e[1]) for e in evs]
    pre_ms = [e[1].elapsed_time(e[2]) for e in evs]
    dec_total = sum(dec_ms)
    pre_total = sum(pre_ms)

    def max_over_ranks(val):
        return reduce_max(val, world, dev)

    total_ms = max_over_ranks(total_ms)
    dec_total = max_over_ranks(dec_total)
    pre_total = max_over_ranks(pre_total)
    dec_avg = dec_total / len(dec_ms)

    # ---------------- context: decode replays back to back, no prefill between
    # (a decode that follows a prefill also writes back the prefill's dirty
    # output lines from L2)
    alone = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
    for a, b_ in alone:
        a.record(stream)
        graphs[0].replay()
        b_.record(stream)
    torch.cuda.synchronize()
    alone_us = sorted(1e3 * a.elapsed_time(b_) for a, b_ in alone)[len(alone) // 2]

    # ---------------- the step beside config 3: variable lengths, contiguous and paged
    extra = None if args.no_extra else measure_varlen(ta, synth, accounting, peaks, dev)
    pi_fig = None if args.no_extra else measure_pi(ta, accounting, peaks, dev, w, q, k, v)
    fp8_fig = None if args.no_extra else measure_fp8(ta, synth, accounting, peaks, dev, w, x)
    nvfp4_fig = None if args.no_extra else measure_nvfp4(ta, synth, accounting, peaks, dev, w, x)
    others_fig = None if args.no_extra else measure_other_configs(ta, synth, accounting, peaks, dev)
    pvar_fig = None if (args.no_extra or not do_prefill) else measure_prefill_varlen(ta, synth, peaks, dev)

    # ---------------- end to end through the public single call, host buffers
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    hq = x["q"].pin_memory()
    hk = x["k"].pin_memory()
    hv = x["v"].pin_memory()
    hout = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16).pin_memory()
    hlse = torch.empty((w.B, w.Hq), dtype=torch.float32).pin_memory()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dws = ta.decode_workspace(w.B, w.Hq, w.Hkv, w.S, w.D, device=dev)

    def e2e_step():
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        ta.decode(dq, dk, dv, scale=w.scale, workspace=dws, out=out, lse=lse)
        hout.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1))
    h2d = hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2
    d2h = hout.numel() * 2 + hlse.numel() * 4

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # ---------------- CPU baseline: the oracle, as it stands, on the host cores
    cpu = None if args.no_cpu_baseline else cpu_baseline_figures(synth, accounting, x)

    dec_s = dec_total / 1e3
    value = replica_throughput(kv_bytes * args.steps, world, dec_s) / 1e9
    achieved = kv_bytes / (dec_avg / 1e3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "accumulate": "f32",
        "data": "synthetic",
        "config": {
            "workload": WORKLOAD_DESC,
            "split_kv": {"n_split": plan.n_split, "chunk": plan.chunk, "grid": plan.grid,
                         "merge": "fused in the decode kernel" if plan.levels == 0
                         else f"{plan.levels} merge launches"},
            "prefill_workload": (f"{PREFILL_WORKLOAD}: B=1, H=32, Hkv=8, D=128, S=16384, causal, bf16"
                                 if do_prefill else "not in this build"),
            "l2": "inputs larger than L2 (512 MiB of K/V per decode step, 335 MB per prefill); no flush",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "us_per_token": round(1e3 * dec_avg, 3),
        "decode_alone": {"us_per_token": round(alone_us, 3),
                         "gbs": round(kv_bytes / (alone_us / 1e6) / 1e9, 1),
                         "frac": round(kv_bytes / (alone_us / 1e6) / 1e9 / peaks["hbm_gbs"], 4),
                         "note": "median of 50 decode replays back to back, after the timed region"},
        "decode_hbm_frac": round(value / world / peaks["hbm_gbs"], 4),
        "roofline": {"bound": "hbm", "kernel": "decode_tc_kernel", "achieved": round(achieved, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": profiled_traffic("decode"), "algorithmic_bytes_per_launch": kv_bytes,
                     "peak_source": peaks["source"] + " (copy bandwidth)",
                     "avg_launch_us": round(1e3 * dec_avg, 3), "launches_per_token": decode_launches},
        "varlen_b16": extra,
        "pi_attention": pi_fig,
        "fp8_kv": fp8_fig,
        "nvfp4_kv": nvfp4_fig,
        "other_decode_configs": others_fig,
        "prefill_varlen": pvar_fig,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "e2e": {"value": round(world * kv_bytes * e2e_steps / (e2e_ms / 1e3) / 1e9, 3), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "call": "ta_decode_ex with pinned host buffers copied in and results copied out"},
        "cpu_baseline": cpu,
    }
    if do_prefill:
        pw = pf[0]
        flops = accounting.prefill_causal_flops(pw.B, pw.Hq, pw.S, pw.D)
        tflops = world * flops * args.steps / (pre_total / 1e3) / 1e12
        line["prefill_tflops"] = round(tflops, 2)
        # the prefill runs in short bursts inside the step (about 2 ms each), at
        # full clocks: the burst peak is its denominator; the sustained one is
        # shown beside it
        line["roofline_prefill"] = {"bound": "tensor", "kernel": "prefill_causal_kernel",
                                    "achieved": round(tflops / world, 2), "peak": peaks["bf16_tflops"],
                                    "unit": "TFLOP/s",
                                    "frac": round(tflops / world / peaks["bf16_tflops"], 4),
                                    "traffic": profiled_traffic("prefill"),
                                    "frac_of_sustained_peak": round(tflops / world / peaks["bf16_tflops_sustained"], 4),
                                    "peak_source": peaks["source"] + " (burst)",
                                    "avg_launch_us": round(1e3 * pre_total / args.steps, 2)}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
