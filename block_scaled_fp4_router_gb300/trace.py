"""Per-phase timeline of the single-launch layer (moe_layer_decode).

    python -m block_scaled_fp4_router_gb300.trace decode1 decode16 batch128 ...

Builds and loads the trace variant of the library (libmoefp4_trace.so,
MOEFP4_TRACE=1), runs a few steps of each workload on one random layer, and
prints, for the last step, when each phase boundary was reached: minimum,
median and maximum over the blocks, in microseconds after the earliest block
started.  With --slots it also prints, per expert slot, when its routed
gate/up and down units were handed out and done and when its h was ready.
The trace stamps are plain stores (per-slot ones: atomics) of %globaltimer, so the timeline
costs the launch a few hundred nanoseconds at most; step times printed here
are host-timed around single launches (no CUDA graph) and are not bench
values.
"""
from __future__ import annotations

import argparse
import os
import statistics

EVENTS = [
    (0, "start"),
    (1, "router done"),
    (3, "x quantised / sorted"),
    (2, "routing built"),
    (4, "sorted x seen (producer)"),
    (5, "shared h seen (producer)"),
    (6, "every routed h seen (producer)"),
    (11, "last shared gate/up unit"),
    (12, "last routed gate/up unit"),
    (13, "last shared down unit"),
    (14, "last routed down unit"),
    (7, "producer done"),
    (8, "units done (epilogue)"),
    (9, "down parts seen"),
    (10, "end (combine done)"),
]


SLOT_COLUMNS = ["gate/up first out", "gate/up last out", "gate/up last done", "h ready", "down first out",
                "down last out", "down last done"]


def slot_table(sl, t0) -> list:
    """Per expert slot: the stamps of its units (us after t0), in slot order."""
    lines = ["| slot | expert | rows | " + " | ".join(SLOT_COLUMNS) + " |", "|---" * (3 + len(SLOT_COLUMNS)) + "|"]
    mask = (1 << 64) - 1
    for s in range(sl.shape[0]):
        info = int(sl[s, 7])
        if info == 0:
            continue
        cells = []
        for c in range(7):
            v = int(sl[s, c])
            if v == 0:
                cells.append("-")
                continue
            if c in (0, 4):  # earliest times are stored complemented
                v = ~v & mask
            cells.append("%.1f" % ((v - t0) / 1e3))
        lines.append("| %d | %d | %d | %s |" % (s, info >> 8, info & 0xFF, " | ".join(cells)))
    return lines


def timeline(name: str, steps: int = 12, device: int = 0, slots: bool = False) -> str:
    import numpy as np
    import torch

    import block_scaled_fp4_router_gb300 as M
    from block_scaled_fp4_router_gb300 import workloads as W
    from block_scaled_fp4_router_gb300.device import DeviceLayer

    wl = W.WORKLOADS[name]
    dev = torch.device("cuda", device)
    lay = DeviceLayer(W.generate_device(wl, 0, dev), wl.H, wl.I, wl.E, wl.top_k, wl.fmt, T_max=wl.T, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    x = torch.randn((wl.T, wl.H), device=dev, generator=gen).to(torch.bfloat16).view(torch.int16)
    b = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    us = []
    for i in range(steps):
        if i == steps - 1:
            torch.cuda.synchronize(dev)
            M.moe_debug_decode_trace(clear=True)
        b.record()
        lay.decode(x)
        e.record()
        torch.cuda.synchronize(dev)
        us.append(b.elapsed_time(e) * 1e3)
    status = M.moe_get_status(lay.ws)
    tr, sl = M.moe_debug_decode_trace(slots=True)
    tr = tr.astype(np.int64)
    started = tr[:, 0] > 0
    t0 = tr[started, 0].min()
    lines = ["%s: T=%d, %d blocks, host-timed step %.1f us (median of %d), status %d"
             % (name, wl.T, int(started.sum()), statistics.median(us[2:]), steps - 2, status),
             "| phase | blocks | min us | median us | max us |", "|---|---|---|---|---|"]
    for ev, label in EVENTS:
        v = tr[:, ev]
        v = v[v > 0]
        if v.size == 0:
            continue
        d = (v - t0) / 1e3
        lines.append("| %s | %d | %.1f | %.1f | %.1f |" % (label, v.size, d.min(), np.median(d), d.max()))
    if slots:
        lines.append("")
        lines += slot_table(sl, int(t0))
    del lay
    torch.cuda.empty_cache()
    return "\n".join(lines)


def main() -> None:
    p = argparse.ArgumentParser()
    p.add_argument("workloads", nargs="+")
    p.add_argument("--steps", type=int, default=12)
    p.add_argument("--slots", action="store_true", help="also a per-slot table of the routed units")
    args = p.parse_args()
    from block_scaled_fp4_router_gb300 import build as B

    B.build(trace=True)
    os.environ["MOEFP4_TRACE"] = "1"
    import block_scaled_fp4_router_gb300 as M

    M.load(M.TRACE_LIB_PATH)
    for name in args.workloads:
        print(timeline(name, args.steps, slots=args.slots))
        print()


if __name__ == "__main__":
    main()
