#!/usr/bin/env python3
"""Benchmark of the paged attention hot path on one GB300 (or N replicas).

One step = one decode step over every layer of the workload: for each layer the
slot write of the new tokens (pa_reshape_and_cache) followed by attention over
the paged cache (pa_decode, or pa_mixed for a mixed batch), all captured in one
CUDA graph.  Inputs are resident in HBM before timing starts.

Printed (rank 0, one JSON line): KV GB/s = algorithmic K/V bytes the step must
read (every cached token of every sequence, every KV head, every layer) divided
by the step time; also sequence-steps/s, the fraction of HBM peak, the
roofline of the dominant kernel (decode; the chunk kernel for a mixed batch),
an end-to-end number through the public API with host buffers, clocks seen
during the timed region, and the CPU oracle's throughput on a bounded sample of
the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_99_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak) and seq-steps/sec"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
DEFAULT_WORKLOAD = "gqa40-8k"
DESCRIPTIONS = {
    "tiny": "tiny decode: 1 layer, B=4, seq_lens 8/17/31/46, H_q=8, H_kv=2, d=128, block 16, bf16",
    "qwen2.5-1.5b": "Qwen2.5-1.5B-shaped decode: 28 layers, B=64, H_q=12, H_kv=2, d=128, block 16, bf16, "
                    "seq_lens~U[512,4096], random block placement",
    "gqa40-8k": "40-layer GQA decode: B=40 at 8192 tokens, H_q=32, H_kv=8, d=128, block 16, fp16 KV",
    "shared-prefix": "shared-prefix decode: 1 layer, B=128, H_q=32, H_kv=8, bf16, 128 aliased prefix blocks "
                     "+ private suffix U[0,1000]",
    "shared-prefix-long": "shared-prefix decode, long prompt: 1 layer, B=32, H_q=32, H_kv=8, bf16, 512 aliased "
                          "prefix blocks (8192 tokens) + private suffix U[0,512]",
    "shared-prefix-l2": "shared-prefix decode, prefix only: 1 layer, B=128, H_q=32, H_kv=8, bf16, 128 aliased "
                        "prefix blocks and no private tokens (the decode's L2 ceiling for shared blocks)",
    "mixed-fp8": "mixed fp8: 1 layer, H_q=64, H_kv=8, e4m3 KV, 16 decode rows (lognormal median 8192, cap 32768) "
                 "+ 2 prefill chunks of 512 on 4096-token contexts",
    "mixed-bf16": "mixed bf16: 1 layer, H_q=64, H_kv=8, bf16 KV, 16 decode rows (lognormal median 8192, cap 32768) "
                  "+ 2 prefill chunks of 512 on 4096-token contexts",
}
ELEM = {"bf16": 2, "fp16": 2, "fp8": 1}


def kv_read_bytes(w: W.Workload) -> int:
    """Algorithmic K/V bytes of one step: 2 * H_kv * d * b per cached token, per layer."""
    return w.num_layers * int(w.seq_lens.sum().item()) * 2 * w.num_kv_heads * w.head_dim * ELEM[w.cache_dtype]


def describe(name: str, block_size: int, num_layers: int | None = None) -> str:
    d = DESCRIPTIONS.get(name, name)
    full = {"qwen2.5-1.5b": 28, "gqa40-8k": 40}.get(name)
    if num_layers is not None and full is not None and num_layers != full:
        d = d.replace(f"{full} layers", f"{num_layers} of {full} layers").replace(
            "40-layer GQA decode", f"40-layer GQA decode ({num_layers} layer{'s' if num_layers > 1 else ''} run)")
    if block_size != W.BLOCK_SIZE:
        d = d.replace("block 16", f"block {block_size}").replace(
            "128 aliased prefix blocks", f"2048-token aliased prefix ({2048 // block_size} blocks of {block_size})").replace(
            "512 aliased prefix blocks", f"{8192 // block_size} aliased prefix blocks of {block_size}")
    return d


def last_block_waste(w: W.Workload) -> float:
    """Share of the allocated cache slots that hold no token: the empty tail of
    every sequence's last block (shared prefix blocks counted once)."""
    bs = w.block_size
    lens = [int(n) for n in w.seq_lens.tolist()]
    pre = w.shared_prefix_blocks * bs
    used = sum(n - pre for n in lens) + (pre if lens else 0)
    alloc = sum(-(-(n - pre) // bs) * bs for n in lens) + (pre if lens else 0)
    return round(1.0 - used / alloc, 5) if alloc else 0.0


def chunk_flops(w: W.Workload) -> int:
    """Algorithmic FLOPs of the prefill chunks of one layer: QK^T and PV, 2 per
    multiply-add, over the causal key range of every chunk row (no padding)."""
    ql = (w.query_start_loc[1:] - w.query_start_loc[:-1]).tolist()
    n = w.seq_lens.tolist()
    keys = sum(q * (n_s - q) + q * (q + 1) // 2 for q, n_s in zip(ql, n) if q > 1)
    return 4 * w.head_dim * w.num_q_heads * keys


def chunk_subbatch(w: W.Workload, layer: int = 0):
    """The chunk rows (q_len > 1) of a mixed batch as a batch of their own."""
    ql = (w.query_start_loc[1:] - w.query_start_loc[:-1]).tolist()
    idx = [i for i, q in enumerate(ql) if q > 1]
    starts = [0]
    for i in idx:
        starts.append(starts[-1] + ql[i])
    dev = w.q[layer].device
    q = torch.cat([w.q[layer][int(w.query_start_loc[i]):int(w.query_start_loc[i + 1])] for i in idx])
    qsl = torch.tensor(starts, dtype=torch.int32, device=dev)
    return q, qsl, w.block_tables[idx].contiguous(), w.seq_lens[idx].contiguous(), max(ql[i] for i in idx)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, world: int) -> float:
    """Max of a float over all ranks (timing only; no data-path collective)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


KERNEL_SOURCES = {"decode": "decode.cu", "chunk": "chunk_tc.cu"}


def kernel_source_hash(kernel: str = "decode") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_99_gb300", "csrc")
    for name in (KERNEL_SOURCES[kernel], "pa_device.cuh", "pa_internal.h"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str = "decode"):
    """DRAM bytes per launch of the workload's decode (or chunk) kernel from a
    committed ncu summary, if it was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(workload)
    if not ent or ent.get("kernel_hash") != kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- our arm

def build_step(w: W.Workload, pa, ws, outs, layers_caches, decode_only_kernels=False, cascade=False,
               before_layer=None, after_layer=None):
    """Enqueue one step on the current stream (used inside graph capture); the optional
    hooks run before and after each layer's calls."""
    for layer in range(w.num_layers):
        if before_layer is not None:
            before_layer(layer)
        enqueue_layer(w, pa, ws, outs, layers_caches, layer, decode_only_kernels, cascade)
        if after_layer is not None:
            after_layer(layer)


def enqueue_layer(w: W.Workload, pa, ws, outs, layers_caches, layer, decode_only_kernels, cascade):
    """Enqueue one layer of the step on the current stream."""
    kc, vc = layers_caches[layer]
    ks = w.k_scale[layer:layer + 1] if w.k_scale is not None else None
    vs = w.v_scale[layer:layer + 1] if w.v_scale is not None else None
    if w.is_decode_only and w.num_new_tokens and not cascade:
        # a decode step: the new tokens' slot write fused into the decode (both graphs)
        pa.pa_decode_append(outs[layer], w.q[layer], w.k_new[layer], w.v_new[layer], w.slot_mapping, kc, vc,
                            w.block_tables, w.seq_lens, w.scale, ws, ks, vs)
        return
    if w.num_new_tokens and not decode_only_kernels:
        pa.pa_reshape_and_cache(w.k_new[layer], w.v_new[layer], kc, vc, w.slot_mapping, ks, vs)
    if w.is_decode_only and cascade:
        pa.pa_decode_shared_prefix(outs[layer], w.q[layer], kc, vc, w.block_tables, w.seq_lens,
                                   w.shared_prefix_blocks, w.scale, ws, ks, vs)
    elif w.is_decode_only:
        pa.pa_decode(outs[layer], w.q[layer], kc, vc, w.block_tables, w.seq_lens, w.scale, ws, ks, vs)
    else:
        pa.pa_mixed(outs[layer], w.q[layer], w.query_start_loc, kc, vc, w.block_tables, w.seq_lens,
                    w.max_q_len, w.scale, ws, ks, vs)


def capture(fn, counted=None):
    """CUDA graph of fn's launches; with `counted` (a list), the number of the
    library's kernels in the graph is appended to it."""
    import paged_kv_cache_99_gb300 as pa
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()          # warm the library's per-device caches outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    before = pa.pa_kernel_launches()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    if counted is not None:
        counted.append(pa.pa_kernel_launches() - before)
    return g


def timed_steps(run_step, steps, min_region_s, est_ms, world):
    """Device time of K steps, repeated in passes until the timed region spans at
    least min_region_s (so that the clock record holds enough samples).  Every
    step is bracketed by its own CUDA events on the launching stream; the region
    by a barrier and a synchronize on both sides.  Returns (ms per step, max over
    ranks), passes, wall seconds of the region."""
    passes = max(1, math.ceil(min_region_s * 1e3 / max(est_ms * steps, 1e-3)))
    passes = int(reduce_max(float(passes), world))
    n = passes * steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n):
        run_step(ev[i])
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier(world)
    ms_local = sum(a.elapsed_time(b) for a, b in ev) / n
    return reduce_max(ms_local, world), passes, wall


def measure(args, name, dev, world, rank, cascade=False, num_layers=None, e2e=True, cpu=False, steps=None):
    """One workload: the step graph timed over the region, the dominant kernel's
    roofline, optionally the end-to-end number and the CPU oracle baseline."""
    import paged_kv_cache_99_gb300 as pa
    steps = steps or args.steps
    kw = {}
    if args.block_size != W.BLOCK_SIZE:
        kw["block_size"] = args.block_size
    if num_layers is not None:
        kw["num_layers"] = num_layers
    w = W.make(name, dev, **kw)
    layers_caches = [(w.k_cache[l], w.v_cache[l]) for l in range(w.num_layers)]
    # the cascade gets the workspace that lets it cut the prefix into key segments
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads, device=dev, shared_prefix=cascade)
    out_all = torch.empty_like(w.q)                      # [layers, rows, H_q, 128]: one buffer
    outs = [out_all[l] for l in range(w.num_layers)]
    kv_bytes = kv_read_bytes(w)
    if cascade and not (w.is_decode_only and w.shared_prefix_blocks > 0):
        raise SystemExit("--cascade needs a decode workload whose tables share leading blocks (shared-prefix)")
    # the library's kernels per step, counted as the step graph is captured
    counted = []
    step_graph = capture(lambda: build_step(w, pa, ws, outs, layers_caches, cascade=cascade), counted)
    decode_graph = capture(lambda: build_step(w, pa, ws, outs, layers_caches, decode_only_kernels=True,
                                              cascade=cascade))
    fused = w.is_decode_only and w.num_new_tokens and not cascade
    launches_per_step = counted[0]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    unique_bytes = sum(c.numel() * c.element_size() * 2 for c in w.k_cache)
    flush = unique_bytes < 2 * l2
    flush_buf = torch.empty(4 * l2, dtype=torch.uint8, device=dev) if flush else None

    def step_with(ev, graph):
        if flush:
            flush_buf.fill_(1)
        ev[0].record()
        graph.replay()
        ev[1].record()

    warm = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.warmup)]
    step_with(warm[0], step_graph)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for e in warm[1:]:
        step_with(e, step_graph)
    torch.cuda.synchronize()
    # wall time per step, L2 flush included: sizes the passes of the timed region
    est_ms = (time.perf_counter() - t0) * 1e3 / max(1, len(warm) - 1)
    status = pa.pa_read_device_status(ws)
    if status != pa.PA_OK:
        raise RuntimeError(f"device status after warm-up: {pa.pa_status_string(status)}")

    # ---- timed region: K steps per pass, passes until the region spans min_region_s ----
    clocks = ClockSampler(int(dev.index or 0))
    ms, passes, t_wall = timed_steps(lambda e: step_with(e, step_graph), steps, args.min_region_s, est_ms, world)
    clk = clocks.stop()

    # ---- the attention calls alone (no separate slot write), same inputs: average call duration ----
    dg_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e in dg_ev:
        step_with(e, decode_graph)
    torch.cuda.synchronize()
    dec_ms = sum(a.elapsed_time(b) for a, b in dg_ev) / steps / w.num_layers

    # ---- a mixed batch is dominated by the chunk kernel: time it on the chunk rows alone ----
    chunk = None
    if not w.is_decode_only:
        cq, cqsl, cbt, csl, cmax = chunk_subbatch(w)
        cws = pa.new_workspace(int(csl.numel()), w.num_q_heads, w.num_kv_heads, device=dev)
        cout = torch.empty_like(cq)
        kc, vc = layers_caches[0]
        ks = w.k_scale[0:1] if w.k_scale is not None else None
        vs = w.v_scale[0:1] if w.v_scale is not None else None
        cg = capture(lambda: pa.pa_mixed(cout, cq, cqsl, kc, vc, cbt, csl, cmax, w.scale, cws, ks, vs))
        for _ in range(3):
            cg.replay()
        cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for e in cev:
            step_with(e, cg)
        torch.cuda.synchronize()
        chunk = (sum(a.elapsed_time(b) for a, b in cev) / steps, chunk_flops(w))

    # ---- end to end through the public API with host buffers ----
    e2e_line = run_e2e(args, w, pa, ws, outs, layers_caches, dev, out_all, cascade, steps) if e2e else None

    peaks, peak_src = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    value = kv_bytes * world / (ms * 1e-3) / 1e9
    per_launch_bytes = kv_bytes / w.num_layers
    if cascade:
        # the cascade reads the shared blocks once: its roofline counts unique bytes
        tok = sum(int(n) - w.shared_prefix_blocks * w.block_size for n in w.seq_lens.tolist())
        tok += w.shared_prefix_blocks * w.block_size
        per_launch_bytes = tok * 2 * w.num_kv_heads * w.head_dim * ELEM[w.cache_dtype]
    achieved = per_launch_bytes / (dec_ms * 1e-3) / 1e9
    # one layer's launch reads the same bytes whatever the number of layers
    traffic = None if cascade else recorded_traffic(name)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.cache_dtype,
        "data": "synthetic",
        "config": {
            "workload": describe(name, w.block_size, w.num_layers),
            "name": name,
            "num_layers": w.num_layers,
            "block_size": w.block_size,
            "last_block_waste": last_block_waste(w),
            "kv_bytes_per_step": kv_bytes,
            "launch": f"one CUDA graph per step: {w.num_layers} x ("
                      + ("pa_decode_append (slot write fused into the decode)" if fused else
                         ("pa_reshape_and_cache + " if w.num_new_tokens else "")
                         + (("pa_decode_shared_prefix" if cascade else "pa_decode") if w.is_decode_only
                            else "pa_mixed")) + ")",
            "l2": ("L2 flushed between steps (a 4 x L2 buffer written before each)" if flush else
                   f"inputs larger than L2 ({unique_bytes / 1e9:.2f} GB of cache vs {l2 / 1e6:.0f} MB L2)"),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "timed_region": {"passes": passes, "steps_timed": passes * steps, "wall_s": round(t_wall, 3),
                         "ms_per_step": "mean over every timed step"},
        "seq_steps_per_s": round(w.num_seqs * world / (ms * 1e-3), 1),
        "pct_of_nominal_hbm": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": round(100 * value / world / hbm_peak, 2),
        "roofline": {
            "kernel": "pa_decode_shared_prefix (unique bytes: prefix once + suffixes)" if cascade else
                      ("pa_decode_append" if fused else
                       ("pa_decode (logical bytes: shared blocks counted per table)" if w.shared_prefix_blocks
                        else "pa_decode")),
            "bound": "hbm",
            "achieved": round(achieved, 2),
            "peak": hbm_peak,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback",
            "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4),
            "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": per_launch_bytes,
            "avg_launch_ms": round(dec_ms, 5),
        },
        "e2e": e2e_line,
        "gpu_launches": launches_per_step * passes * steps,
        "launches_per_step": launches_per_step,
        "clocks": clk,
        "wall_s_timed_region": round(t_wall, 4),
    }
    if chunk is not None:
        # the tensor-core chunk kernel dominates a mixed step: its roofline is the reported one,
        # against the measured dense bf16 rate (f16 runs at the same nominal rate)
        c_ms, c_flops = chunk
        tpeak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
        c_achieved = c_flops / (c_ms * 1e-3) / 1e12
        line["roofline_decode_rows"] = dict(line["roofline"], kernel="pa_mixed (decode rows and chunks)")
        line["roofline"] = {
            "kernel": "chunk_tc (pa_mixed on the chunk rows alone)",
            "bound": "tensor",
            "achieved": round(c_achieved, 2),
            "peak": tpeak,
            "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops, burst)" if peak_src == "measured" else "fallback",
            "unit": "TFLOP/s",
            "frac": round(c_achieved / tpeak, 4),
            "traffic": recorded_traffic(name, "chunk"),
            "algorithmic_flops_per_launch": c_flops,
            "avg_launch_ms": round(c_ms, 5),
        }
    if rank == 0 and cpu:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
        line["cpu_baseline"]["kv_bytes_per_step"] = kv_bytes
    del step_graph, decode_graph, w, layers_caches, ws, out_all, outs, flush_buf
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


# the benchmark spec's targets besides the headline: measured in the same run, each with
# its own timed region and clock record
TARGETS = (("shared-prefix", "shared-prefix", False), ("shared-prefix-cascade", "shared-prefix", True),
           ("mixed-fp8", "mixed-fp8", False))


def target_summary(line):
    keep = ("value", "unit", "ms_per_step", "steps", "seq_steps_per_s", "pct_of_nominal_hbm", "pct_of_measured_hbm",
            "roofline", "roofline_decode_rows", "clocks", "timed_region", "gpu_launches")
    out = {"workload": line["config"]["workload"], "launch": line["config"]["launch"], "l2": line["config"]["l2"],
           "kv_bytes_per_step": line["config"]["kv_bytes_per_step"]}
    out.update({k: line[k] for k in keep if k in line})
    return out


def run_ours(args, rank, world, local):
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    # every replica runs the same workload (weak scaling)
    line = measure(args, args.workload, dev, world, rank, cascade=bool(args.cascade), num_layers=args.layers,
                   e2e=not args.no_e2e, cpu=not args.no_cpu_baseline)
    if not args.no_targets and args.workload == DEFAULT_WORKLOAD and not args.cascade and args.layers is None:
        line["targets"] = {}
        for key, name, casc in TARGETS:
            t = measure(args, name, dev, world, rank, cascade=casc, e2e=False, cpu=False)
            line["targets"][key] = target_summary(t)
    return line


def run_e2e(args, w, pa, ws, outs, layers_caches, dev, out_all, cascade, steps):
    """Same metric through the public API, with the step's inputs copied from pinned
    host memory and the outputs copied back inside the timed region.  The copies run
    on two copy streams beside the attention: the first layer's inputs go first, the
    other layers' inputs follow as one copy per tensor while the first layer is
    attended to (many small copies cost more than their bytes), and each layer's
    output travels back while the next layer runs; the step ends when the last
    output is on the host."""
    per_layer = [w.q, w.k_new, w.v_new]                               # [layers, ...]
    shared = [w.slot_mapping, w.block_tables, w.seq_lens, w.query_start_loc]
    pinned_layer = [t.detach().cpu().pin_memory() for t in per_layer]
    pinned_shared = [t.detach().cpu().pin_memory() for t in shared]
    host_all = torch.empty((len(outs),) + tuple(outs[0].shape), dtype=outs[0].dtype, pin_memory=True)
    host_out = [host_all[l] for l in range(len(outs))]
    h2d = sum(t.numel() * t.element_size() for t in pinned_layer + pinned_shared)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    copy_in, copy_out = torch.cuda.Stream(), torch.cuda.Stream()
    layers = w.num_layers

    def step_calls():
        comp = torch.cuda.current_stream()
        copy_in.wait_stream(comp)
        copy_out.wait_stream(comp)
        first, rest = torch.cuda.Event(), torch.cuda.Event()
        with torch.cuda.stream(copy_in):
            for dst, src in zip(shared, pinned_shared):
                dst.copy_(src, non_blocking=True)
            for dst, src in zip(per_layer, pinned_layer):
                dst[0].copy_(src[0], non_blocking=True)
            first.record(copy_in)
            if layers > 1:
                for dst, src in zip(per_layer, pinned_layer):
                    dst[1:].copy_(src[1:], non_blocking=True)
            rest.record(copy_in)

        def before(layer):
            if layer <= 1:
                comp.wait_event(first if layer == 0 else rest)

        def after(layer):
            # the outputs of all layers but the last go back in one copy while the last
            # layer runs, then the last layer's (outs are the layers of out_all)
            if layer < layers - 2:
                return
            done = torch.cuda.Event()
            done.record(comp)
            copy_out.wait_event(done)
            with torch.cuda.stream(copy_out):
                if layer == layers - 2:
                    host_all[:layers - 1].copy_(out_all[:layers - 1], non_blocking=True)
                else:
                    host_all[layers - 1].copy_(out_all[layers - 1], non_blocking=True)

        build_step(w, pa, ws, outs, layers_caches, cascade=cascade, before_layer=before, after_layer=after)
        comp.wait_stream(copy_out)
        comp.wait_stream(copy_in)

    g = capture(step_calls)
    stream = torch.cuda.current_stream()

    def step():
        g.replay()

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return {"value": round(kv_read_bytes(w) / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


# ----------------------------------------------------------------------------- oracle arm

CODE = {"bf16": 0, "fp16": 1, "fp8": 2}


def raw(t: torch.Tensor) -> np.ndarray:
    """Storage bits of a tensor as numpy (uint16 for 16-bit types, uint8 for FP8)."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


REF_SAMPLE_SEQS = 8


def cpu_baseline(w: W.Workload, seconds: float, total_layers: int | None = None, total_seqs: int | None = None):
    """The oracle as it stands, single-threaded, on a bounded sample of the
    workload: whole layers (slot write + attention for every sequence) until
    `seconds` of oracle time have passed; reported in the same unit (KV GB/s)."""
    import oracle
    per_layer = kv_read_bytes(w) // w.num_layers
    qsl = w.query_start_loc.cpu().numpy()
    tables = w.block_tables.cpu().numpy()
    lens = w.seq_lens.cpu().numpy()
    slots = w.slot_mapping.cpu().numpy()
    elapsed, layers = 0.0, 0
    while layers < w.num_layers and (layers == 0 or elapsed < seconds):
        kc, vc = raw(w.k_cache[layers]), raw(w.v_cache[layers])
        ks = float(w.k_scale[layers]) if w.k_scale is not None else 1.0
        vs = float(w.v_scale[layers]) if w.v_scale is not None else 1.0
        qb = raw(w.q[layers])
        kn, vn = raw(w.k_new[layers]), raw(w.v_new[layers])
        t1 = time.perf_counter()
        if w.num_new_tokens:
            kc, vc = oracle.reshape_and_cache(kn, vn, CODE[w.q_dtype], kc, vc, CODE[w.cache_dtype], slots, ks, vs)
        if w.is_decode_only:
            oracle.decode(qb, CODE[w.q_dtype], kc, vc, CODE[w.cache_dtype], tables, lens, w.scale, ks, vs)
        else:
            oracle.mixed(qb, CODE[w.q_dtype], qsl, kc, vc, CODE[w.cache_dtype], tables, lens, w.scale, ks, vs)
        elapsed += time.perf_counter() - t1
        layers += 1
    return {"value": round(layers * per_layer / elapsed / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{layers} of {total_layers or w.num_layers} layers, "
                      + (f"{w.num_seqs} of {total_seqs} sequences" if total_seqs else "every sequence")
                      + f", slot write + attention, float64, one thread (host has {os.cpu_count()} cores); "
                      "the rate is per KV byte, so it stands for the whole step",
            "seconds": round(elapsed, 3)}


def run_reference(args, rank, world):
    """The oracle on the host cores, same workload, metric and unit; each step a
    bounded sample (whole layers)."""
    if rank != 0:
        return None
    kw = {"num_layers": 1} if args.workload in ("qwen2.5-1.5b", "gqa40-8k") else {}
    if args.workload == "gqa40-8k":
        kw["batch"] = REF_SAMPLE_SEQS       # a sample of the 40 equal sequences: the rate is per byte
    if args.block_size != W.BLOCK_SIZE:
        kw["block_size"] = args.block_size
    w = W.make(args.workload, "cpu", **kw)
    total = {"qwen2.5-1.5b": 28, "gqa40-8k": 40}.get(args.workload, w.num_layers)
    seqs = {"gqa40-8k": 40}.get(args.workload)
    per_step = []
    for _ in range(args.warmup + args.steps):
        per_step.append(cpu_baseline(w, args.ref_step_seconds, total, seqs))
    timed = per_step[args.warmup:]
    value = statistics.mean(x["value"] for x in timed)
    ms = statistics.mean(1e3 * x["seconds"] for x in timed)
    cb = dict(timed[-1])
    cb["value"] = round(value, 4)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(args.workload, w.block_size), "name": args.workload,
                   "block_size": w.block_size},
        "cpu_baseline": cb,
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_copy_blocks(args, rank, world, local):
    """Copy-on-write block copies (pa_copy_blocks) on a pool shaped like one layer of the
    40-layer GQA model (8 KV heads, fp16): `pairs` distinct src -> dst blocks per step."""
    import paged_kv_cache_99_gb300 as pa
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    nb, hkv, pairs = 40_000, 8, 16_384
    g = torch.Generator(device=dev).manual_seed(1010)
    bs = args.block_size
    nb = nb * W.BLOCK_SIZE // bs                         # the same pool and copied bytes at every block size
    pairs = pairs * W.BLOCK_SIZE // bs
    k = torch.randn(nb, hkv, bs, 128, generator=g, device=dev).half()
    v = torch.randn(nb, hkv, bs, 128, generator=g, device=dev).half()
    perm = torch.randperm(nb, generator=g, device=dev).int()
    src, dst = perm[:pairs].contiguous(), perm[pairs:2 * pairs].contiguous()
    block_bytes = hkv * bs * 128 * 2
    moved = 2 * pairs * block_bytes * 2                  # K and V, read + write
    for _ in range(args.warmup):
        pa.pa_copy_blocks(k, v, src, dst)
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        ev[i][0].record()
        pa.pa_copy_blocks(k, v, src, dst)
        ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = reduce_max(sum(a.elapsed_time(b) for a, b in ev) / args.steps, world)
    peaks, peak_src = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    gbs = moved / (ms * 1e-3) / 1e9
    return {
        "metric": "copy-on-write block copy GB/s (read + write bytes)",
        "value": round(gbs * world, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp16", "data": "synthetic",
        "config": {"workload": f"copy {pairs} blocks of {hkv} KV heads x {bs} x 128 fp16 (K and V) per step, "
                               f"pool of {nb} blocks ({2 * nb * block_bytes / 1e9:.1f} GB)",
                   "l2": "inputs larger than L2"},
        "roofline": {"kernel": "copy_blocks_kernel", "bound": "hbm", "achieved": round(gbs, 2), "peak": hbm_peak,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, a copy)", "unit": "GB/s",
                     "frac": round(gbs / hbm_peak, 4), "traffic": None, "algorithmic_bytes_per_launch": moved,
                     "avg_launch_ms": round(ms, 5)},
        "gpu_launches": args.steps, "clocks": clk,
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.NAMED))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cascade", action="store_true",
                    help="shared-prefix workload through pa_decode_shared_prefix (prefix once on the tensor cores)")
    ap.add_argument("--op", default="attention", choices=["attention", "copy-blocks"],
                    help="copy-blocks: time the copy-on-write block copies instead of the attention step")
    ap.add_argument("--block-size", type=int, default=W.BLOCK_SIZE, choices=[8, 16, 32],
                    help="tokens per cache block (the named workloads are built with 16)")
    ap.add_argument("--layers", type=int, default=None,
                    help="run only this many layers of a multi-layer workload (e.g. 1 for an ncu capture)")
    ap.add_argument("--no-targets", action="store_true",
                    help="skip the shared-prefix, cascade and mixed-fp8 measurements that follow the default headline")
    ap.add_argument("--min-region-s", type=float, default=2.5,
                    help="repeat the K timed steps in passes until the timed region spans this many seconds")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=4.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    elif args.op == "copy-blocks":
        line = run_copy_blocks(args, rank, world, local)
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
