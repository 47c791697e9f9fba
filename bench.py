#!/usr/bin/env python
"""Benchmark of the block-scaled FP4 MoE layer on GB300.

One step = one pass of the whole layer (router, top-k, MXFP4 activation
quantisation, permutation, routed SwiGLU experts with the requantise
epilogue, BF16 shared expert, weighted combine) over one batch of synthetic
tokens.  The default workload is the 1-row decode layer (H=4096, I=1536,
128 MXFP4 experts, top-4, BF16 shared expert), run through the fused
single-launch decode entry point.

Timing: steps are captured in a CUDA graph (S steps per graph, replayed R
times, K = R*S) so that host launch overhead does not enter; every step uses
a different layer of 8 distinct weight sets (about 10.6 GB, far above the
129 MB L2) and a fresh token row.  The timed graph holds only the steps; a
second graph with a CUDA event pair around every step, replayed after the
timed region, gives the per-step kernel durations for the roofline, which
counts the bytes the step must read: the touched experts' FP4 codes and
scales, the shared expert, the router and the token rows.

`--impl reference` times the CPU oracle on the host cores on the same
workload (a bounded sample of steps).

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s; decode expert-weight HBM GB/s; prefill FP4 TFLOPS vs peak"
N_LAYERS = 8


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=6000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="decode1")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-budget-s", type=float, default=15.0)
    p.add_argument("--layers", type=int, default=N_LAYERS,
                   help="distinct weight sets rotated over the steps (8 keeps inputs far above L2)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def expert_bytes(wl) -> int:
    """FP4 codes + scales of one routed expert (gate, up and down)."""
    per_scale = 16 if wl.fmt == "nvfp4" else 32
    w13 = 2 * wl.I * wl.H // 2 + 2 * wl.I * wl.H // per_scale
    w2 = wl.H * wl.I // 2 + wl.H * wl.I // per_scale
    ts = 12 if wl.fmt == "nvfp4" else 0
    return w13 + w2 + ts


def step_bytes(wl, n_distinct: int) -> int:
    """Algorithmic bytes of one decode step: touched experts + shared expert +
    router (+ bias) + token rows in and out."""
    # the shared expert: BF16, or one more FP4 expert when folded into the table
    shared = expert_bytes(wl) if wl.shared_fp4 else (3 * wl.H * wl.I * 2 if wl.shared else 0)
    router = wl.E * wl.H * 4 + (wl.E * 4 if wl.zipf > 0 else 0)
    return n_distinct * expert_bytes(wl) + shared + router + 2 * wl.T * wl.H * 2


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
                "samples": len(rows)}


# ------------------------------------------------------------- CPU oracle


def oracle_rate(wl, budget_s: float, max_steps: int):
    """Times the oracle on steps of the workload (T tokens each) on layer 0
    until the budget is spent; returns (tokens/s, steps, tokens, seconds)."""
    from block_scaled_fp4_router_gb300 import workloads as W
    from oracle import moe as O

    lay = W.generate(wl)
    t0 = time.perf_counter()
    steps = 0
    while steps < max_steps:
        xs = W.generate_tokens(wl, 1000 + steps, wl.T)
        step_layer = dict(lay)
        step_layer["x"] = xs
        O.layer_forward(step_layer, wl.top_k, wl.fmt)
        steps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return wl.T * steps / dt, steps, wl.T * steps, dt


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
    wl = W.WORKLOADS[args.workload]
    budget = max(10.0, min(120.0, 12.0 * max(1, args.steps) ** 0.5))
    oracle_rate(wl, 1e-9, max(0, min(args.warmup, 1)))  # warm-up: one step
    rate, steps, toks, dt = oracle_rate(wl, budget, args.steps)
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * dt / max(steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(wl), "parallelism": "replicas"},
        "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": "%d of %d steps (%d tokens) of the workload on the host cores, "
                                   "float64 numpy oracle" % (steps, args.steps, toks)},
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



def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import block_scaled_fp4_router_gb300 as pkg
    from block_scaled_fp4_router_gb300 import build as B
    from block_scaled_fp4_router_gb300 import workloads as W
    from block_scaled_fp4_router_gb300.device import DeviceLayer

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

    wl = W.WORKLOADS[args.workload]
    fused = wl.T <= 16
    T, K, Wm = wl.T, max(1, args.steps), max(3, args.warmup)
    # graph of S steps replayed R times, S a divisor of K
    S = max(d for d in range(1, min(K, 256) + 1) if K % d == 0)
    R = K // S
    nl = max(1, args.layers)
    layers = [DeviceLayer(W.generate_device(wl, l + 97 * rank, dev), wl.H, wl.I, wl.E, wl.top_k, wl.fmt,
                          T_max=T, device=dev) for l in range(nl)]
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    xs = (torch.randn((S, T, wl.H), device=dev, generator=gen)).to(torch.bfloat16).view(torch.int16)
    outs = [layers[i % nl].outputs(T) for i in range(S)]
    stream = torch.cuda.Stream(device=dev)

    def step(i):
        lay = layers[i % nl]
        if fused:
            lay.decode(xs[i], *outs[i])
        else:
            lay.forward(xs[i], *outs[i])

    # layers, inputs and outputs were made on the default stream
    stream.wait_stream(torch.cuda.current_stream(dev))
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(Wm):  # untimed warm-up steps
            step(i % S)
    torch.cuda.synchronize(dev)
    # The timed graph holds only the steps; a second graph with an event pair
    # around every step gives the per-step kernel durations for the roofline
    # (event nodes between the kernels would otherwise stretch the step time).
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(S):
            step(i)
    ev = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
          for _ in range(S)]
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=stream):
        for i in range(S):
            ev[i][0].record()
            step(i)
            ev[i][1].record()
    graph.replay()  # graph warm-up (not timed)
    torch.cuda.synchronize(dev)
    st = pkg.moe_get_status(layers[0].ws)
    if st != pkg.MOE_OK:
        raise RuntimeError("device status after warm-up: %s" % pkg.moe_status_string(st))

    # ---- timed region: exactly K steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler()
    clocks.start()
    time.sleep(0.3)  # let the sampler come up
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record()
        for _ in range(R):
            graph.replay()
        t1.record()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    phys = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").replace(",", "").isdigit() else local
    clk = clocks.stop(phys)
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    for lay in layers:
        st = pkg.moe_get_status(lay.ws)
        if st != pkg.MOE_OK:
            raise RuntimeError("device status after the timed region: %s" % pkg.moe_status_string(st))

    # ---- per-step kernel durations and the bytes each step needed
    with torch.cuda.stream(stream):
        graph_ev.replay()
        graph_ev.replay()
    torch.cuda.synchronize(dev)
    durs = np.array([ev[i][0].elapsed_time(ev[i][1]) * 1e-3 for i in range(S)])  # seconds
    distinct = np.array([len(np.unique(outs[i][1].cpu().numpy())) for i in range(S)])
    byts = np.array([step_bytes(wl, int(n)) for n in distinct], dtype=np.float64)
    achieved = float(byts.sum() / durs.sum() / 1e9)
    peak, peak_kind = peaks()

    # ---- end to end through the public API with host buffers: every step
    # copies its x from pinned host memory, runs the layer and copies out back
    # to pinned host memory, all captured in a CUDA graph as a serving engine
    # runs its decode steps (no Python in the timed loop)
    S_e = min(S, 250)
    R_e = max(1, min(K, 500) // S_e)
    n_e2e = S_e * R_e
    x_host = torch.empty((S_e, T, wl.H), dtype=torch.int16, pin_memory=True)
    x_host.copy_(xs[torch.arange(S_e, device=dev) % S].cpu())
    out_host = torch.empty((S_e, T, wl.H), dtype=torch.int16, pin_memory=True)
    x_dev = torch.empty((T, wl.H), dtype=torch.int16, device=dev)
    o_dev, i_dev, w_dev = layers[0].outputs(T)
    torch.cuda.synchronize(dev)

    def e2e_step(i):
        # H2D and D2H through the library's SM copy (moe_copy_rows)
        pkg.moe_copy_rows(x_dev, x_host[i])
        lay = layers[i % nl]
        (lay.decode if fused else lay.forward)(x_dev, o_dev, i_dev, w_dev)
        pkg.moe_copy_rows(out_host[i], o_dev)

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
    e2e_ms = e0.elapsed_time(e1)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle runs after every GPU measurement, on this process's host cores
        rate, steps, toks, dt = oracle_rate(wl, args.cpu_budget_s, 10 ** 6)
        cpu = {"value": rate, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": "%d steps (%d tokens) of the workload's layer 0 in %.1f s, float64 numpy oracle "
                         "(BLAS on all cores)" % (steps, toks, dt)}

    if rank != 0:
        return
    value = replica_throughput(ms, world, T, K)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "mxfp4" if wl.fmt == "mxfp4" else "nvfp4", "data": "synthetic",
        "config": {"workload": describe(wl), "entry_point": "moe_layer_decode" if fused else "moe_layer_forward",
                   "tokens_per_step": T, "layers_rotated": nl,
                   "l2": "inputs larger than L2: %d distinct layers (%.1f GB) rotated every step" % (
                       nl, nl * step_bytes(wl, wl.E) / 1e9),
                   "graph": "%d replays of a %d-step CUDA graph" % (R, S), "parallelism": "replicas"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": NCU_TRAFFIC.get((wl.name, "k_decode_tc")) if fused and layers[0].prepared else None,
                     "peak_kind": peak_kind,
                     "kernel": ("k_decode_tc" if layers[0].prepared and wl.H % 256 == 0 and wl.I % 256 == 0
                                else "k_fused_decode") if fused else "unfused sequence",
                     "kernel_us": float(durs.mean() * 1e6),
                     "bytes_per_step": float(byts.mean()), "distinct_experts_per_step": float(distinct.mean())},
        "e2e": {"value": T * n_e2e / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": T * wl.H * 2,
                "d2h_bytes_per_step": T * wl.H * 2, "steps": n_e2e,
                "graph": "%d replays of a %d-step CUDA graph of (H2D x, layer, D2H out), the copies by "
                         "moe_copy_rows from / to pinned host memory" % (R_e, S_e)},
        "gpu_launches": K if fused else None,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


# dram__bytes_read.sum + dram__bytes_write.sum of one launch, from the ncu
# capture summarised in profiles/k_decode_tc_decode1.md (same kernel source).
NCU_TRAFFIC = {("decode1", "k_decode_tc"): 82.00e6}


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
