#!/usr/bin/env python
"""Benchmark of the routed MoE layer stack with the LRU expert cache.

One step = one batch of T tokens through every layer of the stack, the whole
hot path per layer: router logits, softmax/top-k, permutation, device LRU, miss
copies from the pinned host banks, SwiGLU experts and combine. Default
workload: decode T=1 on the 40-layer NVFP4 stack (H=2048, E=256, k=8, I=512,
Zipf s=1.0 routing) with a pool of 25% of all experts; every step draws fresh
seeded hidden states for each layer. The default line also carries a
``prefill`` object: T=4096 on the first 4 layers of the 40-layer BF16 stack,
once with every expert resident and once with a pool of 50% and next-layer
prefetch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|decode8|prefill|large|large_prefill|stress|decode_fp8|prefill_fp8]

Three passes run over the same step sequence, each from the same cache state
(the pool is rebuilt and the same W warm-up steps run first): the timed pass
(no instrumentation: ``value``), the end-to-end pass through host buffers
(``e2e``) and a pass with per-kernel CUDA events (``kernels_us_per_call``,
``roofline``). Prints one JSON line. --impl reference times the oracle (plain
single-threaded CPU) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s (decode T=1, prefill T=4096); % of HBM / FP4 tensor roofline"
UNIT = "tokens/s"

WORKLOADS = {
    # name: (shape, T, pool fraction, cache flags, layers used, step reuse probability)
    "decode": (synth.DECODE_NVFP4, 1, 0.25, 0, 40, 0.0),
    "decode8": (synth.DECODE_NVFP4, 8, 0.25, 0, 40, 0.0),
    "prefill": (synth.PREFILL_BF16, 4096, 0.5, 1, 40, 0.0),
    "large": (synth.LARGE_MXFP4, 1, 0.2, 0, 24, 0.0),
    "large_prefill": (synth.LARGE_MXFP4, 2048, 0.2, 0, 24, 0.0),
    "stress": (synth.STRESS_NVFP4, 1, 0.10, 0, 16, 0.7),
    "decode_fp8": (synth.DECODE_FP8, 1, 0.25, 0, 40, 0.0),
    "prefill_fp8": (synth.PREFILL_FP8, 4096, 0.5, 1, 40, 0.0),
}

PREFILL_LAYERS = 4  # layers of the prefill stack in the default line's prefill object


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


def host_info():
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
    except Exception:
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.device = device
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.device), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx = max(mx, float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic_for(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source has not changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[f"{kernel}/{workload}"]
        if e["source_hash"] != _source_hash(e["sources"]):
            return None
        return e["dram_bytes_per_launch"]
    except Exception:
        return None


# --------------------------------------------------------------------------- replicas

def rank_hidden_states(shape, rank, nsteps, L, T, reuse):
    """Hidden states [nsteps, L, T, H] (bf16 bits) of one rank. Every rank
    draws its own steps (replicas share no inputs); with step reuse, a step
    repeats the previous step's hidden states in every layer."""
    hid = np.empty((nsteps, L, T, shape.H), np.uint16)
    flags_r = synth.reuse_flags(rank, nsteps, reuse) if reuse > 0 else np.zeros(nsteps, bool)
    src = 0
    for st in range(nsteps):
        src = src if flags_r[st] else st
        for l in range(L):
            hid[st, l] = synth.hidden_states(shape, 0, l, T, step=1000003 * rank + src)
    return hid


def max_over_ranks(dist, x, device=None):
    """The largest x over all ranks (x itself without a process group). NCCL
    reduces a device tensor, gloo a host tensor."""
    if not dist:
        return float(x)
    import torch
    on_dev = dist.get_backend() == "nccl"
    t = torch.tensor([float(x)], dtype=torch.float64, device=device if on_dev else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, steps, T, ms_max):
    """Whole-job tokens/s: every rank runs `steps` steps of T tokens of its own;
    the job takes as long as its slowest rank."""
    return world * steps * T / (ms_max * 1e-3)


# --------------------------------------------------------------------------- our arm

def load_stack(moe, shape, L, capacity, flags, device, max_tokens, seed=0):
    desc = moe.make_desc(L, shape.E, shape.k, shape.H, shape.I, shape.fmt, shape.act, shared=shape.shared,
                         mode=shape.act_mode, max_tokens=max_tokens, device=device)
    h = moe.moe_init(desc)

    def load_layer(l):
        for e in range(shape.E + shape.shared):
            moe.moe_load_expert(h, l, e, synth.expert_weights(shape, seed, l, e))

    with ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        list(ex.map(load_layer, range(L)))
    moe.moe_cache_config(h, capacity, flags)
    return h


def h2d_peak_gbs(torch, device, nbytes=1 << 30, reps=10):
    """Best of `reps` pinned host -> device cudaMemcpyAsync of nbytes, timed
    with CUDA events on the copy's stream."""
    from cuda.bindings import runtime as cudart
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s = torch.cuda.Stream(device=device)
    best = 0.0
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        err, = cudart.cudaMemcpyAsync(dst.data_ptr(), src.data_ptr(), nbytes,
                                      cudart.cudaMemcpyKind.cudaMemcpyHostToDevice, s.cuda_stream)
        if err != cudart.cudaError_t.cudaSuccess:
            raise RuntimeError(f"cudaMemcpyAsync: {err}")
        b.record(s)
        s.synchronize()
        best = max(best, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    del src, dst
    return best


def run_passes(moe, torch, h, shape, L, T, S, flags, hid, router, dev, W, K, dist, sample_clocks=True, prewarm=None):
    """The three passes over steps 0..W+K-1 of `hid` (numpy [steps, L, T, H]),
    each after rebuilding the pool (same cache state) and the same W warm-up
    steps: timed (no instrumentation), end to end (host buffers), per-kernel
    timing. Returns the measurements."""
    x_dev = torch.from_numpy(hid.view(np.int16)).to(dev).view(torch.bfloat16)
    out_dev = torch.empty((L, T, shape.H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream

    # device pointers of every call, taken before the timed regions (a caller of
    # the C ABI holds raw pointers; tensor indexing is not part of the call)
    r_ptr = [router[l].data_ptr() for l in range(L)]
    o_ptr = [out_dev[l].data_ptr() for l in range(L)]
    x_ptr = [[x_dev[st, l].data_ptr() for l in range(L)] for st in range(hid.shape[0])]
    fwd = moe.load().moe_layer_forward  # the C entry point; errors surface at moe_sync

    def step(st, ptrs):
        xp = ptrs[st]
        for l in range(L):
            rc = fwd(h, xp[l], r_ptr[l], l, T, o_ptr[l], sp)
            if rc:
                moe.moe_sync(h)  # raises the call's error
                raise RuntimeError(f"moe_layer_forward returned {rc}")

    def fresh():
        moe.moe_cache_config(h, S, flags)
        if prewarm is not None:
            prewarm(stream)
        for st in range(W):
            step(st, x_ptr)
        moe.moe_sync(h)
        stream.synchronize()
        moe.moe_stats_reset(h)

    # ---- timed pass
    fresh()
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    clocks = ClockSampler(dev.index) if sample_clocks else None
    if clocks:
        clocks.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    hw0 = time.perf_counter()
    for st in range(W, W + K):
        step(st, x_ptr)
    host_ms = (time.perf_counter() - hw0) * 1e3 / K  # enqueue time per step (host-bound if close to ms_per_step)
    ev1.record(stream)
    stream.synchronize()
    moe.moe_sync(h)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(dist, ev0.elapsed_time(ev1), dev)
    stats = moe.moe_stats(h)

    # ---- end to end through host buffers, same steps from the same cache state
    hid_pin = torch.from_numpy(hid.view(np.int16)).view(torch.bfloat16).pin_memory()
    out_pin = torch.empty((L, T, shape.H), dtype=torch.bfloat16).pin_memory()
    xin = torch.empty((L, T, shape.H), dtype=torch.bfloat16, device=dev)
    xin_ptr = [[xin[l].data_ptr() for l in range(L)]]
    fresh()
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    e0.record(stream)
    for st in range(W, W + K):
        with torch.cuda.stream(stream):
            xin.copy_(hid_pin[st], non_blocking=True)
        step(0, xin_ptr)
        with torch.cuda.stream(stream):
            out_pin.copy_(out_dev, non_blocking=True)
        stream.synchronize()
    e1.record(stream)
    stream.synchronize()
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1), dev)
    e2e_wall = (time.perf_counter() - w0) * 1e3
    e2e_stats = moe.moe_stats(h)

    # ---- per-kernel CUDA events, same steps from the same cache state
    fresh()
    moe.moe_timing_enable(h, True)
    for st in range(W, W + K):
        step(st, x_ptr)
    moe.moe_sync(h)
    timing = moe.moe_timing(h)
    moe.moe_timing_enable(h, False)
    del x_dev, hid_pin, out_pin, xin
    return {"ms": ms, "e2e_ms": e2e_ms, "e2e_wall": e2e_wall, "timing": timing, "stats": stats,
            "e2e_misses": e2e_stats["misses"], "clk": clk, "host_ms": host_ms}


def prefill_object(moe, torch, dev, args):
    """Prefill workload T=4096 on the first PREFILL_LAYERS layers of the BF16
    stack: every expert resident, then a pool of 50% with next-layer prefetch."""
    shape, T = synth.PREFILL_BF16, 4096
    L = PREFILL_LAYERS
    W, K = 2, 3
    t0 = time.time()
    full = L * shape.E
    h = load_stack(moe, shape, L, full, 0, dev.index, max_tokens=T)
    load_s = time.time() - t0
    router = [torch.from_numpy(synth.router_weights(shape, 0, l).view(np.int16)).to(dev).view(torch.bfloat16)
              for l in range(L)]
    hid = rank_hidden_states(shape, 0, W + K, L, T, 0.0)
    blob = moe.moe_expert_bytes(moe.make_desc(1, shape.E, shape.k, shape.H, shape.I, shape.fmt, shape.act))
    res = {}
    for name, S, flags in (("resident", full, 0), ("pool_50pct_prefetch", full // 2, moe.MOE_CACHE_PREFETCH_NEXT_LAYER)):
        m = run_passes(moe, torch, h, shape, L, T, S, flags, hid, router, dev, W, K, None, sample_clocks=False)
        res[name] = (S, flags, m)
    moe.moe_destroy(h)
    return {"shape": shape, "T": T, "L": L, "W": W, "K": K, "load_s": load_s, "blob": blob, "passes": res,
            "cpu": cpu_baseline(shape, T, 40, budget_s=args.cpu_budget / 2) if args.cpu_budget > 0 else None}


def run_ours(args, rank, world, dist):
    import torch
    import expert_offload_softmax_b300 as moe
    from expert_offload_softmax_b300 import build
    build.build()
    moe.load()
    local = _env_int("LOCAL_RANK", 0)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    shape, T, frac, flags, L, reuse = WORKLOADS[args.workload]
    if args.sync_misses:
        flags |= moe.MOE_CACHE_SYNC_MISSES
    if args.host_misses:
        flags |= moe.MOE_CACHE_HOST_MISSES
    if args.layers:
        L = min(L, args.layers)
    if args.pool_frac:
        frac = args.pool_frac
    if args.resident:
        frac = 1.0
    cap_shape = synth.Shape("cap", L=L, E=shape.E, k=shape.k, H=shape.H, I=shape.I, fmt=shape.fmt, act=shape.act)
    S = synth.capacity_slots(cap_shape, frac)
    t_load = time.time()
    Tw = 4096  # resident mode: one call of this many tokens per layer loads every expert
    h = load_stack(moe, shape, L, S, flags, local, max_tokens=max(T, Tw if args.resident else 8))
    t_load = time.time() - t_load
    router = [torch.from_numpy(synth.router_weights(shape, 0, l).view(np.int16)).to(dev).view(torch.bfloat16)
              for l in range(L)]
    hid = rank_hidden_states(shape, rank, args.warmup + args.steps, L, T, reuse)
    prewarm = None
    if args.resident:
        xw = torch.from_numpy(synth.hidden_states(shape, 0, 0, Tw, step=999983).view(np.int16)).to(dev).view(torch.bfloat16)
        ow = torch.empty((Tw, shape.H), dtype=torch.bfloat16, device=dev)

        def prewarm(stream):
            for l in range(L):
                moe.moe_layer_forward(h, xw.data_ptr(), router[l].data_ptr(), l, Tw, ow.data_ptr(), stream.cuda_stream)
            moe.moe_sync(h)
            stream.synchronize()
    meas = run_passes(moe, torch, h, shape, L, T, S, flags, hid, router, dev, args.warmup, args.steps, dist,
                      prewarm=prewarm)
    moe.moe_destroy(h)
    blob = moe.moe_expert_bytes(moe.make_desc(1, shape.E, shape.k, shape.H, shape.I, shape.fmt, shape.act,
                                              shared=shape.shared))
    if rank != 0:
        return None
    meas.update({"pcie": h2d_peak_gbs(torch, dev), "t_load": t_load, "S": S, "frac": frac, "flags": flags, "L": L,
                 "resident": bool(args.resident)})
    pre = None
    if world == 1 and args.workload == "decode" and args.prefill_object:
        pre = prefill_object(moe, torch, dev, args)
    line = make_line(args, world, meas, blob)
    if pre is not None:
        line["prefill"] = prefill_section(pre)
    return line


def _kernel_us(timing):
    calls = max(1, timing["resident_calls"])
    return {"route+cache": round(timing["route_ms"] * 1e3 / max(1, timing["calls"]), 2),
            "gate_up": round(timing["gate_up_ms"] * 1e3 / calls, 2),
            "down": round(timing["down_ms"] * 1e3 / calls, 2),
            "combine": round(timing["combine_ms"] * 1e3 / calls, 2),
            "resident_calls": int(timing["resident_calls"]), "calls": int(timing["calls"])}


def _tensor_roofline(shape, T, timing, peaks, peak_kind, which="gate_up"):
    """The prefill expert GEMM as a dense contraction: gate/up is 2*2*I*H flops
    per routed row, down 2*H*I."""
    calls = max(1, timing["resident_calls"])
    rows = T * (shape.k + shape.shared)
    flops = (4.0 if which == "gate_up" else 2.0) * shape.I * shape.H * rows
    ms = timing[f"{which}_ms"] / calls
    tf = flops / (ms * 1e-3) / 1e12 if ms > 0 else 0.0
    tpeak = peaks.get("bf16_tflops", 1800.0)
    nbytes = timing[f"{which}_bytes"] / calls
    gbs = nbytes / (ms * 1e-3) / 1e9 if ms > 0 else 0.0
    hpeak = peaks.get("hbm_gbs", 6400.0)
    return {"bound": "tensor", "kernel": ("gate/up + SwiGLU" if which == "gate_up" else "down projection")
            + " grouped GEMM (tcgen05, TMA, TMEM)",
            "achieved": round(tf, 1), "peak": tpeak, "unit": "TFLOP/s", "frac": round(tf / tpeak, 4),
            "peak_source": f"{peak_kind} bf16_tflops (MEASURED_PEAKS.json)",
            "algorithmic_flops_per_launch": flops, "avg_launch_us": round(ms * 1e3, 3),
            "hbm": {"algorithmic_bytes_per_launch": int(nbytes), "achieved_gbs": round(gbs, 1),
                    "frac": round(gbs / hpeak, 4)}}


def prefill_section(pre):
    peaks, peak_kind = _peaks()
    shape, T, L, K = pre["shape"], pre["T"], pre["L"], pre["K"]
    out = {"workload": shape.name, "T": T, "layers": L, "steps": K, "warmup": pre["W"],
           "load_s": round(pre["load_s"], 1), "cpu_baseline": pre["cpu"]}
    for name, (S, flags, m) in pre["passes"].items():
        timing, stats = m["timing"], m["stats"]
        d = {"pool_slots": S, "cache_flags": flags, "value": round(K * T / (m["ms"] * 1e-3), 1), "unit": UNIT,
             "ms_per_step": round(m["ms"] / K, 3),
             "kernels_us_per_call": _kernel_us(timing),
             "cache": {"misses_per_step": round(stats["misses"] / K, 2),
                       "prefetch_misses_per_step": round(stats["prefetch_misses"] / K, 2),
                       "h2d_bytes_per_step": int(stats["bytes_h2d"] // K)},
             "miss_stream_gbs": round(timing["copy_bytes"] / (timing["copy_ms"] * 1e-3) / 1e9, 2)
             if timing["copy_ms"] > 0 else None}
        if timing["resident_calls"] > 0:
            d["roofline"] = _tensor_roofline(shape, T, timing, peaks, peak_kind, "gate_up")
            d["roofline_down"] = _tensor_roofline(shape, T, timing, peaks, peak_kind, "down")
        out[name] = d
    return out


def _dtype_str(fmt, T):
    """The arithmetic the path computes in, for the JSON line's dtype."""
    if fmt == synth.FMT_BF16:
        return "bf16 x bf16, fp32 accumulate"
    if fmt == synth.FMT_FP32:
        return "fp32"
    wide = "f16" if T <= 8 else "bf16"
    w = {synth.FMT_NVFP4: "nvfp4 weights (E2M1 code x E4M3 block scale, exact in %s)" % wide,
         synth.FMT_MXFP4: "mxfp4 weights (E2M1 code exact in %s, E8M0 block scale %s)" % (
             wide, "in fp32 per 32-element partial sum" if T <= 8 else "folded in, exact in bf16"),
         synth.FMT_FP8: "fp8 weights (E4M3 code exact in %s, per-tensor scale after the dot product)" % wide}[fmt]
    act = ("activations scaled by a power of two per token row into f16" if T <= 8 else "bf16 activations")
    return w + " x " + act + ", fp32 accumulate"


def make_line(args, world, meas, blob_bytes):
    """The bench's JSON line from one run's measurements: meas holds the timed
    and end-to-end durations (ms, max over ranks), the library's timing and
    stats counters, the PCIe peak, the clock record and the run's stack
    parameters; blob_bytes is one expert's size in the device layout."""
    shape, T, _, _, _, reuse = WORKLOADS[args.workload]
    ms, e2e_ms, e2e_wall = meas["ms"], meas["e2e_ms"], meas["e2e_wall"]
    timing, stats, pcie, clk, t_load = meas["timing"], meas["stats"], meas["pcie"], meas["clk"], meas["t_load"]
    S, frac, flags, L = meas["S"], meas["frac"], meas["flags"], meas["L"]
    blob = blob_bytes
    peaks, peak_kind = _peaks()
    K = args.steps
    value = job_value(world, K, T, ms)
    # dominant library kernel by device time, over the calls without demand
    # misses (a call with misses also waits for its copies inside the kernel)
    kern = {"gate_up": (timing["gate_up_ms"], timing["gate_up_bytes"]),
            "down": (timing["down_ms"], timing["down_bytes"])}
    if timing["combine_ms"] > 0:
        kern["combine"] = (timing["combine_ms"], timing["combine_bytes"])
    fused_decode = T <= 8 and shape.fmt in (synth.FMT_NVFP4, synth.FMT_MXFP4, synth.FMT_FP8)
    if fused_decode:
        # one kernel does the whole call: routing, cache lookup, gate/up, down, combine
        kern = {"gate_up": (timing["gate_up_ms"], timing["gate_up_bytes"] + timing["down_bytes"])}
    dom = max(kern, key=lambda n: kern[n][0])
    dms, dbytes = kern[dom]
    calls = max(1, timing["resident_calls"])
    kernel_name = {"gate_up": "k_decode (router, top-k, cache lookup, gate/up, down, combine)"
                   if fused_decode else "gate/up + SwiGLU",
                   "down": "down projection", "combine": "combine"}[dom]
    achieved = dbytes / (dms * 1e-3) / 1e9 if dms > 0 else 0.0
    peak = peaks.get("hbm_gbs", 6400.0)
    traffic = _traffic_for("k_decode" if fused_decode else dom, args.workload)
    roof = {"bound": "hbm", "kernel": kernel_name, "achieved": round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4),
            "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
            else "fallback 6.4 TB/s",
            "algorithmic_bytes_per_launch": int(dbytes // calls),
            "avg_launch_us": round(dms * 1e3 / calls, 3),
            "traffic": traffic}
    if T > 8:
        roof = _tensor_roofline(shape, T, timing, peaks, peak_kind, "gate_up")
        roof["traffic"] = traffic
    cpu = cpu_baseline(shape, T, L, budget_s=args.cpu_budget) if world == 1 else None
    ws_bytes = (stats["hits"] + stats["misses"]) * blob // max(1, K)
    cap_hits = stats["hits"] + stats["misses"]
    dev_copies = T <= 8 and shape.fmt in (synth.FMT_NVFP4, synth.FMT_MXFP4, synth.FMT_FP8) and not (flags & 8)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms / K, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": _dtype_str(shape.fmt, T),
        "data": "synthetic (seeded; random weights of the stated shape)",
        "config": {"workload": shape.name,
                   "T": T, "layers": L, "pool_slots": S, "pool_frac": frac,
                   "router_zipf_s": shape.zipf_s, "cache_flags": flags, "step_reuse_p": reuse,
                   "shared_experts": shape.shared,
                   "miss_copies": "decode kernel reads the mapped pinned banks" if dev_copies
                   else "host cudaMemcpyAsync on a side stream",
                   "cache_state": ("every expert resident: each pass rebuilds the pool, loads every expert "
                                   "with one 4096-token call per layer, then runs the warm-up steps")
                   if meas.get("resident") else "each pass rebuilds the pool and runs the same warm-up steps first",
                   "l2": "per-step working set (the weights of every expert a step selects, %d MB) exceeds "
                         "the 126 MB L2" % (ws_bytes // (1 << 20)),
                   "parallelism": "replicas" if world > 1 else "1 GPU"},
        "roofline": roof,
        "kernels_us_per_call": _kernel_us(timing),
        "h2d_copy_ms_per_step": round(timing["copy_ms"] / K, 4),
        "host_enqueue_ms_per_step": round(meas.get("host_ms", 0.0), 4),
        "cache": {"hit_rate": round(stats["hits"] / cap_hits, 4) if cap_hits else None,
                  "misses_per_step": round(stats["misses"] / K, 3),
                  "h2d_bytes_per_step": int(stats["bytes_h2d"] // K),
                  "prefetch_misses_per_step": round(stats["prefetch_misses"] / K, 3)},
        "pcie": {"h2d_peak_gbs": round(pcie, 2),
                 "h2d_peak_method": "best of 10 x 1 GiB pinned cudaMemcpyAsync, CUDA events",
                 "miss_stream_gbs": round(timing["copy_bytes"] / (timing["copy_ms"] * 1e-3) / 1e9, 2)
                 if timing["copy_ms"] > 0 else None},
        "e2e": {"value": round(world * K * T / (e2e_ms * 1e-3), 3), "unit": UNIT,
                "h2d_bytes_per_step": L * T * shape.H * 2, "d2h_bytes_per_step": L * T * shape.H * 2,
                "wall_ms": round(e2e_wall, 2), "misses_per_step": round(meas.get("e2e_misses", 0) / K, 3)},
        "gpu_launches": int(stats["kernel_launches"]),
        "load_s": round(t_load, 1),
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    return line


# --------------------------------------------------------------------------- oracle

ORACLE_TOKEN_SAMPLE = 16  # above this many tokens a call is timed on samples
ORACLE_DEQUANT_SAMPLE = 2  # experts dequantised per sampled call
ORACLE_PAIR_SAMPLE = 8     # (token, expert) products per sampled call


def oracle_call_seconds(shape, T, L, layer, step, lru, routers):
    """Seconds of one oracle layer call (T tokens, layer `layer`, hidden states
    of `step`). Up to ORACLE_TOKEN_SAMPLE tokens the whole call is timed:
    routing, LRU, dequantisation of the selected experts and the layer's expert
    math. Above it (prefill; one call of the large stack takes many minutes on
    one core, most of it dequantising 257 experts) each part is timed on a
    sample and scaled to the full call: routing of evenly spaced tokens by
    T / tokens, dequantisation of a few selected experts to every expert of the
    layer (a prefill call of T*k >= 8*E assignments selects them all), and the
    expert FFN on a few (token, expert) pairs to all T*(k + shared) pairs.
    Expert weights are generated untimed. Returns (seconds, tokens routed)."""
    import oracle
    from moe_harness import act_to_f32
    if layer not in routers:
        routers[layer] = act_to_f32(synth.router_weights(shape, 0, layer), shape)
    sampled = T > ORACLE_TOKEN_SAMPLE
    ns = ORACLE_TOKEN_SAMPLE if sampled else T
    toks = np.linspace(0, T - 1, ns).round().astype(np.int64)
    shared = list(range(shape.E, shape.E + shape.shared))
    x = act_to_f32(synth.hidden_states(shape, 0, layer, T, step=step), shape)[toks]
    t0 = time.perf_counter()
    r = oracle.route(x, routers[layer], shape.k)
    lru.access(layer, r["uniq"], T, False)
    t1 = time.perf_counter()
    need = sorted(set(int(e) for e in np.unique(r["topk_idx"])) | set(shared))
    if sampled:
        need = need[:ORACLE_DEQUANT_SAMPLE]
    raw = {e: synth.expert_weights(shape, 0, layer, e) for e in need}
    t2 = time.perf_counter()
    ws = {e: oracle.dequant_expert(shape.fmt, raw[e], shape.H, shape.I) for e in need}
    t3 = time.perf_counter()
    if sampled:
        for i in range(ORACLE_PAIR_SAMPLE):
            oracle.expert_ffn(x[i % ns], *ws[need[i % len(need)]], shape.act_mode)
    else:
        oracle.layer_tokens(x, r["topk_idx"], r["gates"], ws, shape.E, shape.shared, shape.act_mode, np.arange(ns))
    t4 = time.perf_counter()
    if sampled:
        est = ((t1 - t0) * T / ns + (t3 - t2) * (shape.E + shape.shared) / len(need)
               + (t4 - t3) * T * (shape.k + shape.shared) / ORACLE_PAIR_SAMPLE)
    else:
        est = (t1 - t0) + (t4 - t2)
    return est, ns


def oracle_layer_seconds(shape, T, L, budget_s, step0=0):
    """Oracle layer calls of the workload (T tokens, cycling through the
    layers) until ~budget_s of oracle time has elapsed; at least one call.
    Returns (mean seconds per full layer call, calls, tokens routed per call)."""
    import oracle
    lru = oracle.LRU(L, shape.E, max(shape.E, synth.capacity_slots(shape, 0.25)))
    routers = {}
    spent, total, calls, ns = 0.0, 0.0, 0, T
    while spent < budget_s or calls == 0:
        t0 = time.perf_counter()
        est, ns = oracle_call_seconds(shape, T, L, calls % L, step0 + calls, lru, routers)
        spent += time.perf_counter() - t0
        total += est
        calls += 1
    return total / calls, calls, ns


def _sample_note(shape, T, ns):
    if ns >= T:
        return ""
    return (f"; each call timed on samples scaled to the full call: routing of {ns} evenly spaced "
            f"tokens, dequantisation of {ORACLE_DEQUANT_SAMPLE} of the {shape.E + shape.shared} "
            f"experts, the expert FFN on {ORACLE_PAIR_SAMPLE} of the {T * (shape.k + shape.shared)} "
            f"(token, expert) pairs")


def cpu_baseline(shape, T, L, budget_s=15.0):
    if budget_s <= 0:
        return None
    per_call, calls, ns = oracle_layer_seconds(shape, T, L, budget_s)
    sample = (f"{calls} layer calls (T={T}) of the {L}-layer stack; tokens/s = T / (L x mean s per call)"
              + _sample_note(shape, T, ns))
    return {"value": round(T / (per_call * L), 4), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
            **host_info()}


def run_reference(args):
    """The oracle as it stands, on the host cores: each step is one oracle layer
    call of the workload (cycling through the stack's layers), timed whole up to
    16 tokens, on samples above; tokens/s = T / (L x mean seconds per call),
    i.e. the stack's rate at the measured per-layer cost."""
    import oracle
    shape, T, frac, flags, L, reuse = WORKLOADS[args.workload]
    cap_shape = synth.Shape("cap", L=L, E=shape.E, k=shape.k, H=shape.H, I=shape.I, fmt=shape.fmt, act=shape.act)
    S = synth.capacity_slots(cap_shape, frac)
    lru = oracle.LRU(L, shape.E, max(shape.E, S))
    routers = {}
    for w in range(args.warmup):
        oracle_call_seconds(shape, T, L, w % L, w, lru, routers)
    secs, ns = [], T
    t_run = time.perf_counter()
    for st in range(args.steps):
        i = args.warmup + st
        s_call, ns = oracle_call_seconds(shape, T, L, i % L, i, lru, routers)
        secs.append(s_call)
    run_s = time.perf_counter() - t_run
    ms = float(np.mean(secs)) * 1e3
    value = T / (L * ms * 1e-3)
    sample = (f"{args.steps} timed oracle layer calls (T={T}, cycling through the {L} layers) after "
              f"{args.warmup} untimed ones; tokens/s = T / ({L} x mean s per call)" + _sample_note(shape, T, ns))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "step": "one oracle layer call of the stack (the GPU arm's step runs every layer)",
        "timed_s": round(run_s, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32 (CPU oracle)",
        "data": "synthetic (seeded; random weights of the stated shape)",
        "config": {"workload": shape.name, "T": T, "layers": L, "pool_slots": S, "pool_frac": frac,
                   "router_zipf_s": shape.zipf_s, "cache_flags": flags, "step_reuse_p": reuse,
                   "shared_experts": shape.shared, "parallelism": "1 GPU"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                         **host_info()},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default 100 decode, 3 prefill)")
    ap.add_argument("--warmup", type=int, default=None, help="warm-up steps (default 20 decode, 3 prefill)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--layers", type=int, default=0, help="run only the first N layers of the stack (profiling)")
    ap.add_argument("--sync-misses", action="store_true",
                    help="service each host-copied miss before the call's expert kernels are launched "
                         "(for profilers that serialise launches; not a bench setting)")
    ap.add_argument("--host-misses", action="store_true",
                    help="decode: copy misses with cudaMemcpyAsync from the host instead of from the kernel")
    ap.add_argument("--no-prefill-object", dest="prefill_object", action="store_false",
                    help="leave the prefill measurement out of the default decode line")
    ap.add_argument("--pool-frac", type=float, default=0.0,
                    help="expert pool as a fraction of the stack's experts (default: the workload's)")
    ap.add_argument("--resident", action="store_true",
                    help="resident-only phase: a pool of every expert, each loaded before the warm-up, so no "
                         "timed call misses")
    args = ap.parse_args()
    decode = WORKLOADS[args.workload][1] <= 8
    if args.steps is None:
        args.steps = 100 if decode else 3
    if args.warmup is None:
        args.warmup = 20 if decode else 3
    if args.warmup < 3:
        args.warmup = 3
    rank = _env_int("RANK", 0)
    world = _env_int("WORLD_SIZE", 1)
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(_env_int("LOCAL_RANK", 0))
        tdist.init_process_group("nccl")
        dist = tdist
    line = run_ours(args, rank, world, dist)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
