#!/usr/bin/env python
"""Benchmark of the block-scaled FP4 MoE layer on GB300.

One step = one pass of the whole layer (router, top-k, MXFP4 activation
quantisation, permutation, routed SwiGLU experts with the requantise
epilogue, the shared expert, weighted combine) over one batch of synthetic
tokens.  The headline workload is the 8192-token prefill layer (H=4096,
I=1536, 128 MXFP4 experts, top-4 under a Zipf(1.1) router bias, BF16 shared
expert) through moe_layer_forward; the other layer workloads (tiny, 1-token
decode, 16-token NVFP4 decode uniform and Zipf(1.2), the 128-token batch
through moe_layer_forward and, as "batch128@decode", through the
single-launch moe_layer_decode (also with an MXFP8 shared expert), the
prefill with an MXFP8 shared expert) are
measured in the same run under "per_config".

Timing (every workload): S steps are captured in a CUDA graph and replayed R
times, so that one timed region is exactly K = R * S steps; the region is
timed with CUDA events on the launching stream and repeated until the regions
add up to at least 1 s; the median region gives the value, min / max the
spread.  Every step uses one of 8 distinct weight sets (at least 0.9 GB
each, far above the 129 MB L2) and its own token rows.  A second graph with
event nodes around every step (and, for the prefill, around its two routed
FP4 GEMMs) is replayed after the timed regions for per-step durations.

Rooflines: the prefill's routed gate/up + down GEMMs against the FP4 tensor
peak (2 T k 3 H I FLOP per step over their event-timed duration); the decode
workloads against the measured HBM copy bandwidth on the bytes a step must
read (touched experts' FP4 codes and scales, the shared expert, the router,
token rows in and out) over the timed per-step time.

`--impl reference` times the CPU oracle on the host cores on the headline
workload (a bounded sample per step).

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s; decode expert-weight HBM GB/s; prefill FP4 TFLOPS vs peak"
N_LAYERS = 8
# "name@decode": the workload through moe_layer_decode (one launch) whatever its size
PER_CONFIG = ["tiny", "decode1", "decode16", "decode16z", "batch128", "batch128@decode", "batch128_s8@decode",
              "prefill8k_s8"]
# nominal dense GB300 tensor rates (PFLOP/s): FP4 13.5, BF16 2.25
FP4_PER_BF16 = 13.5 / 2.25
MIN_REGION_S = 1.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="prefill8k",
                   help="the headline workload (name@decode: through moe_layer_decode, one launch)")
    p.add_argument("--configs", default=",".join(PER_CONFIG),
                   help="workloads measured under per_config (comma list, '' for none)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-budget-s", type=float, default=10.0)
    p.add_argument("--min-region-s", type=float, default=MIN_REGION_S)
    p.add_argument("--layers", type=int, default=N_LAYERS,
                   help="distinct weight sets rotated over the steps (8 keeps inputs far above L2)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "kind": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "kind": "fallback"}


def expert_bytes(wl) -> int:
    """FP4 codes + scales of one routed expert (gate, up and down)."""
    per_scale = 16 if wl.fmt == "nvfp4" else 32
    w13 = 2 * wl.I * wl.H // 2 + 2 * wl.I * wl.H // per_scale
    w2 = wl.H * wl.I // 2 + wl.H * wl.I // per_scale
    ts = 12 if wl.fmt == "nvfp4" else 0
    return w13 + w2 + ts


def step_bytes(wl, n_distinct: int) -> int:
    """Algorithmic bytes of one step: touched experts + shared expert +
    router (+ bias) + token rows in and out."""
    # the shared expert: BF16, or one more FP4 expert when folded into the table
    shared = expert_bytes(wl) if wl.shared_fp4 else (3 * wl.H * wl.I * 2 if wl.shared else 0)
    router = wl.E * wl.H * 4 + (wl.E * 4 if wl.zipf > 0 else 0)
    return n_distinct * expert_bytes(wl) + shared + router + 2 * wl.T * wl.H * 2


def routed_flop(wl) -> float:
    """FLOP of the routed gate/up and down contractions of one step."""
    return 2.0 * wl.T * wl.top_k * 3 * wl.H * wl.I


def largest_divisor(K: int, cap: int) -> int:
    return max(d for d in range(1, max(1, min(K, cap)) + 1) if K % d == 0)


# ------------------------------------------------------------------ clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "100",
                 "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, gpu_index=0):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for ln in f:
                    parts = [p.strip() for p in ln.split(",")]
                    if len(parts) >= 9 and parts[0].isdigit() and int(parts[0]) == gpu_index:
                        rows.append(parts)
            os.unlink(self.path)
        except Exception:
            return None
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = sorted(float(r[1]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows)}


# ------------------------------------------------------------- CPU oracle

PREFILL_SLICE = 512  # tokens per oracle step on the prefill workload


def oracle_rate(wl, budget_s: float, max_steps: int):
    """Times the oracle on the workload's layer 0 on the host cores: one
    untimed warm-up step, then steps of fresh token rows (the whole batch, or
    a PREFILL_SLICE-token slice of the prefill batch) until the budget is
    spent.  The oracle's expert cache is shared across the steps (each expert
    dequantised once, as a layer kept resident on the CPU).  Returns
    (tokens/s, steps, tokens, seconds, sample description)."""
    from block_scaled_fp4_router_gb300 import workloads as W
    from oracle import moe as O

    T = min(wl.T, PREFILL_SLICE)
    lay = W.generate(wl, tokens=T)
    cache = {}

    def one(seed):
        step_layer = dict(lay)
        step_layer["x"] = W.generate_tokens(wl, seed, T)
        O.layer_forward(step_layer, wl.top_k, wl.fmt, cache=cache)

    one(999)  # warm-up (fills the expert cache for the experts it touches)
    t0 = time.perf_counter()
    steps = 0
    while steps < max(1, max_steps):
        one(1000 + steps)
        steps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    what = ("%d steps of %d tokens (%s) on the host cores after one untimed warm-up step, float64 numpy "
            "oracle with its expert cache shared across steps" % (
                steps, T, "a %d-token slice of the %d-token batch" % (T, wl.T) if T < wl.T else "the whole batch",))
    del cache, lay
    gc.collect()
    return T * steps / dt, steps, T * steps, dt, what


def describe(wl):
    return ("%s: T=%d tokens/step, H=%d, I=%d, E=%d routed top-%d %s + %s, seed %d%s" % (
        wl.name, wl.T, wl.H, wl.I, wl.E, wl.top_k, wl.fmt.upper(),
        "%s shared expert folded into the table" % wl.fmt.upper() if wl.shared_fp4 else
        ("BF16 shared expert" if wl.shared else "no shared expert"), wl.seed,
        ", Zipf(%.1f) router bias" % wl.zipf if wl.zipf else ""))


def run_reference(args):
    from block_scaled_fp4_router_gb300 import workloads as W

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = W.WORKLOADS[args.workload.partition("@")[0]]
    budget = max(10.0, min(120.0, 12.0 * max(1, args.steps) ** 0.5))
    rate, steps, toks, dt, what = oracle_rate(wl, budget, args.steps)
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * dt / max(steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(wl), "parallelism": "replicas"},
        "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": "%s (%d of the %d requested steps fit the %.0f s budget)" % (
                             what, steps, args.steps, budget)},
        "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- our kernels


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest replica's timed-region length: every rank calls this after
    its own timing (a collective when world > 1)."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(ms: float, world: int, T: int, K: int) -> float:
    """Whole-job tokens/s of `world` independent replicas, each stepping T
    tokens K times, over the slowest replica's time (weak scaling)."""
    return world * T * K / (ms * 1e-3)


def measure(wl, args, dev, rank, world, pk, headline: bool, entry=None):
    """One workload: timed regions of exactly K steps, per-step durations,
    roofline, end to end through the C ABI from host buffers, clocks."""
    import numpy as np
    import torch
    import torch.distributed as dist

    import block_scaled_fp4_router_gb300 as pkg
    from block_scaled_fp4_router_gb300 import workloads as W
    from block_scaled_fp4_router_gb300.device import DeviceLayer

    fused = entry == "decode" if entry else wl.T <= 16
    T, K, Wm = wl.T, max(1, args.steps), max(3, args.warmup)
    # a graph of S steps replayed R times; S divides K and the S steps' token
    # rows and outputs stay within about 2 GB
    S = largest_divisor(K, min(256, max(1, int(2e9 // (T * wl.H * 4)))))
    R = K // S
    nl = max(1, args.layers)
    layers = [DeviceLayer(W.generate_device(wl, l + 97 * rank, dev), wl.H, wl.I, wl.E, wl.top_k, wl.fmt,
                          T_max=T, device=dev) for l in range(nl)]
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    xs = torch.randn((S, T, wl.H), device=dev, generator=gen).to(torch.bfloat16).view(torch.int16)
    outs = [layers[i % nl].outputs(T) for i in range(S)]
    stream = torch.cuda.Stream(device=dev)

    def step(i, x=None, o=None):
        lay = layers[i % nl]
        x = xs[i] if x is None else x
        o = outs[i] if o is None else o
        (lay.decode if fused else lay.forward)(x, *o)

    stream.wait_stream(torch.cuda.current_stream(dev))
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(Wm):  # untimed warm-up steps
            step(i % S)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    n0 = pkg.moe_debug_launch_count()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(S):
            step(i)
    launches_per_step = (pkg.moe_debug_launch_count() - n0) / S
    # per-step event pairs (and, on the batched path, the routed GEMMs' pair)
    ev = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
          for _ in range(S)]
    gev = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
           for _ in range(S)]
    with torch.cuda.stream(stream):  # torch creates an event at its first record: before its handle is passed on
        for pair in gev:
            for e in pair:
                e.record()
    torch.cuda.synchronize(dev)
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=stream):
        for i in range(S):
            pkg.moe_set_timing_events(*gev[i])
            ev[i][0].record()
            step(i)
            ev[i][1].record()
    pkg.moe_set_timing_events(None, None)
    graph.replay()  # graph warm-up (not timed)
    torch.cuda.synchronize(dev)
    for lay in layers:
        st = pkg.moe_get_status(lay.ws)
        if st != pkg.MOE_OK:
            raise RuntimeError("%s: device status after warm-up: %s" % (wl.name, pkg.moe_status_string(st)))

    # ---- timed regions, each exactly K steps, until they add up to >= min_region_s
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler()
    clocks.start()
    time.sleep(0.3)  # let the sampler come up
    regions = []
    while sum(regions) < 1000.0 * args.min_region_s or len(regions) < 3:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t0.record()
            for _ in range(R):
                graph.replay()
            t1.record()
        torch.cuda.synchronize(dev)
        regions.append(t0.elapsed_time(t1))
        if len(regions) >= 100000:
            break
    if world > 1:
        dist.barrier()
    phys = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(dev.index)).split(",")[dev.index]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").replace(",", "").isdigit() else dev.index
    clk = clocks.stop(phys)
    ms = max_over_ranks(statistics.median(regions), world, dev)
    for lay in layers:
        st = pkg.moe_get_status(lay.ws)
        if st != pkg.MOE_OK:
            raise RuntimeError("%s: device status after the timed regions: %s" % (wl.name, pkg.moe_status_string(st)))

    # ---- per-step durations from the event graph
    with torch.cuda.stream(stream):
        graph_ev.replay()
        graph_ev.replay()
    torch.cuda.synchronize(dev)
    step_us = np.array([ev[i][0].elapsed_time(ev[i][1]) * 1e3 for i in range(S)])
    distinct = np.array([len(np.unique(outs[i][1].cpu().numpy())) for i in range(S)])
    byts = np.array([step_bytes(wl, int(n)) for n in distinct], dtype=np.float64)
    ms_step = ms / K
    res = {
        "workload": describe(wl),
        "entry_point": ("moe_layer_decode" if fused else "moe_layer_forward")
        + ("_shared_mxfp8" if wl.shared and wl.shared_fmt == "mxfp8" else ""),
        "tokens_per_step": T, "value": replica_throughput(ms, world, T, K), "unit": "tokens/s",
        "ms_per_step": ms_step, "steps": K,
        "timing": {"regions": len(regions), "region_ms_median": statistics.median(regions),
                   "region_ms_min": min(regions), "region_ms_max": max(regions),
                   "timed_s": sum(regions) / 1e3,
                   "graph": "%d replays of a %d-step CUDA graph per region" % (R, S),
                   "step_us_event_graph": float(step_us.mean())},
        "gpu_launches_per_step": launches_per_step,
        "clocks": clk,
    }
    hbm = {"bound": "hbm", "achieved": float(byts.mean() / (ms_step * 1e-3) / 1e9), "peak": pk["hbm_gbs"],
           "unit": "GB/s", "peak_kind": pk["kind"], "traffic": None,
           "bytes_per_step": float(byts.mean()), "distinct_experts_per_step": float(distinct.mean()),
           "time_basis": "timed per-step time (median region / K)"}
    hbm["frac"] = hbm["achieved"] / hbm["peak"]
    if fused:
        prep = layers[0].prepared and wl.H % 256 == 0 and wl.I % 256 == 0
        hbm["kernel"] = ("k_decode_tc (wide step)" if wl.T > 16 else "k_decode_tc") if prep else "k_fused_decode"
        res["roofline"] = hbm
    else:
        hbm["kernel"] = "the layer's launch sequence"
        try:  # recorded only when the routed experts ran on tensor cores
            gemm_us = np.array([gev[i][0].elapsed_time(gev[i][1]) * 1e3 for i in range(S)])
        except RuntimeError:
            gemm_us = None
        fp4 = None
        if gemm_us is not None:
            flop = routed_flop(wl)
            peak = pk["bf16_tflops"] * FP4_PER_BF16
            ach = flop / (gemm_us.mean() * 1e-6) / 1e12
            fp4 = {
                "bound": "tensor", "pipe": "fp4 (kind::mxf4)", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "traffic": None, "peak_kind": pk["kind"],
                "peak_derivation": "%.1f TFLOP/s = %.0f x the measured BF16 burst %.1f TFLOP/s (nominal dense "
                                   "GB300 FP4 : BF16 = 13.5 : 2.25)" % (peak, FP4_PER_BF16, pk["bf16_tflops"]),
                "frac_of_sustained_peak": ach / (pk["bf16_tflops_sustained"] * FP4_PER_BF16),
                "kernel": "routed gate/up + down GEMMs (event-timed together)",
                "flop_per_step": flop, "gemm_us": float(gemm_us.mean()),
                "gemm_share_of_step": float(gemm_us.mean() / (ms_step * 1e3)),
            }
        # the prefill is a contraction: its headline roofline is the FP4 pipe;
        # the batched decode streams its weights: HBM
        if headline and fp4 is not None:
            res["roofline"] = fp4
            res["layer_hbm"] = hbm
        else:
            res["roofline"] = hbm
            if fp4 is not None:
                res["routed_gemms_fp4"] = fp4

    # ---- end to end through the C ABI with host buffers: every step copies
    # its x from pinned host memory, runs the layer and copies out back to
    # pinned host memory (moe_copy_rows), captured in a CUDA graph
    S_e = largest_divisor(K, min(250, max(1, int(5e8 // (T * wl.H * 4)))))
    R_e = K // S_e
    x_host = torch.empty((S_e, T, wl.H), dtype=torch.int16, pin_memory=True)
    x_host.copy_(xs[torch.arange(S_e, device=dev) % S].cpu())
    out_host = torch.empty((S_e, T, wl.H), dtype=torch.int16, pin_memory=True)
    x_dev = torch.empty((T, wl.H), dtype=torch.int16, device=dev)
    o_dev = layers[0].outputs(T)
    torch.cuda.synchronize(dev)

    def e2e_step(i):
        pkg.moe_copy_rows(x_dev, x_host[i])
        step(i, x_dev, o_dev)
        pkg.moe_copy_rows(out_host[i], o_dev[0])

    with torch.cuda.stream(stream):
        for i in range(min(Wm, S_e)):
            e2e_step(i)
    torch.cuda.synchronize(dev)
    graph_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_e2e, stream=stream):
        for i in range(S_e):
            e2e_step(i)
    graph_e2e.replay()  # not timed
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(R_e):
            graph_e2e.replay()
        e1.record()
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    res["e2e"] = {"value": replica_throughput(e2e_ms, world, T, K), "unit": "tokens/s",
                  "h2d_bytes_per_step": T * wl.H * 2, "d2h_bytes_per_step": T * wl.H * 2, "steps": K,
                  "graph": "%d replays of a %d-step CUDA graph of (H2D x, layer, D2H out), the copies by "
                           "moe_copy_rows from / to pinned host memory" % (R_e, S_e)}
    res["inputs"] = "%d distinct layers (%.1f GB of expert weights) rotated every step: inputs larger than " \
                    "L2" % (nl, nl * step_bytes(wl, wl.E) / 1e9)
    del graph, graph_ev, graph_e2e, layers, xs, outs, x_host, out_host
    gc.collect()
    torch.cuda.empty_cache()
    return res


def cpu_baseline(wl, budget_s):
    rate, steps, toks, dt, what = oracle_rate(wl, budget_s, 10 ** 6)
    return {"value": rate, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle", "sample": what}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import block_scaled_fp4_router_gb300 as pkg
    from block_scaled_fp4_router_gb300 import build as B
    from block_scaled_fp4_router_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        B.build()
    if world > 1:
        dist.barrier()
    pkg.load()
    pk = peaks()

    head_name, _, head_entry = args.workload.partition("@")
    wl = W.WORKLOADS[head_name]
    head = measure(wl, args, dev, rank, world, pk, headline=True, entry=head_entry or None)
    per = {}
    for name in [c for c in args.configs.split(",") if c and c != args.workload]:
        base, _, entry = name.partition("@")
        per[name] = measure(W.WORKLOADS[base], args, dev, rank, world, pk, headline=False, entry=entry or None)

    # the oracle runs after every GPU measurement, on this process's host cores
    if rank == 0 and not args.no_cpu_baseline:
        head["cpu_baseline"] = cpu_baseline(wl, args.cpu_budget_s)
        done = {}  # one oracle timing per workload, whatever the entry point
        for name in per:
            base = name.partition("@")[0]
            if base not in done:
                done[base] = cpu_baseline(W.WORKLOADS[base], args.cpu_budget_s / 2)
            per[name]["cpu_baseline"] = done[base]
    if rank != 0:
        return
    K = head["steps"]
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.fmt, "data": "synthetic",
        "config": {"workload": head["workload"], "entry_point": head["entry_point"], "tokens_per_step": wl.T,
                   "l2": head["inputs"], "graph": head["timing"]["graph"], "parallelism": "replicas"},
        "timing": head["timing"],
        "roofline": head["roofline"],
        "e2e": head["e2e"],
        "gpu_launches": int(round(head["gpu_launches_per_step"] * K)),
        "clocks": head["clocks"],
        "cpu_baseline": head.get("cpu_baseline"),
        "per_config": per,
    }
    if "layer_hbm" in head:
        line["layer_hbm"] = head["layer_hbm"]
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
