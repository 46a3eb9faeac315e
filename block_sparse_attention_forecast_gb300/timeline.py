"""Per-CTA timeline of the decode step's per-layer launches (a diagnostic, not the product).

    python -m block_sparse_attention_forecast_gb300.timeline [--layers 6] [--batch 16]

Builds the timeline variant of the library (libsparda_timeline.so, compiled with
-DSPARDA_TIMELINE: every CTA of attend-and-score and of the decode prologue records
%globaltimer at entry, after its wait for the previous launch where it waits, and at exit),
runs a resident stack of `layers` layers at context 131072 in the pipelined layout from a CUDA
graph, and prints, per layer, the phases of the critical path in microseconds relative to the
release of the layer's prologue top-k:

  topk_end     last top-k CTA of the prologue exits (the layer's blocks are known)
  proj         first start and last end of the prologue's projection CTAs
  score_start  first selection CTA of the layer's attend-and-score starts
  attn_end     last attention CTA exits;  sel_end: last selection CTA exits
  next_release the next prologue's top-k CTAs are released (the launch has completed)

The workload is the benchmark's, with fewer layers (seeded synthetic K/V, 16 planted blocks).
"""
from __future__ import annotations

import argparse
import ctypes
import os
import sys

import numpy as np

ROLE = {1: "attention", 2: "selection", 3: "projection", 4: "topk", 5: "append"}


class Rec(ctypes.Structure):
    _fields_ = [("t_entry", ctypes.c_uint64), ("t_release", ctypes.c_uint64), ("t_exit", ctypes.c_uint64),
                ("launch", ctypes.c_uint32), ("role_cta", ctypes.c_uint32)]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--layers", type=int, default=6)
    ap.add_argument("--batch", type=int, default=16)
    args = ap.parse_args()
    from block_sparse_attention_forecast_gb300 import build
    os.environ["SPARDA_LIB"] = build.build(timeline=True)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import torch
    import bench
    import block_sparse_attention_forecast_gb300.binding as sb
    read = sb.lib.sparda_timeline_read
    read.restype = ctypes.c_int32
    read.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32), ctypes.c_int32]
    if args.batch != bench.BATCH:
        bench.BATCH = args.batch
    shape, stack, T0 = bench.build_workload("cuda:0", 0, 4, args.layers, "pipelined")
    stack.advance = False
    stack.capture()
    for _ in range(3):
        stack.run()
    torch.cuda.synchronize()
    n = ctypes.c_int32(0)
    read(None, 0, ctypes.byref(n), 1)                # clear what the warm-up recorded
    stack.run()
    torch.cuda.synchronize()
    cap = 1 << 16
    buf = (Rec * cap)()
    assert read(ctypes.addressof(buf), cap, ctypes.byref(n), 1) == 0
    recs = buf[:n.value]
    t_base = min(r.t_entry for r in recs)
    by_launch = {}
    for r in recs:
        by_launch.setdefault(r.launch, []).append(r)
    launches = sorted(by_launch)
    # launch order per step: score(layer 0, the separate forecast_score launch is not recorded),
    # then per layer L: prologue(L), attend_and_score(L) (layer L < n-1)
    rows = []
    for lid in launches:
        rs = by_launch[lid]
        roles = {ROLE[r.role_cta >> 24] for r in rs}
        kind = "prologue" if roles & {"topk", "projection", "append"} else "attend"
        rows.append((lid, kind, rs))
    us = lambda t: (t - t_base) / 1e3
    print("launch  kind      span (us from the replay's first record)")
    layer_phases = []
    for lid, kind, rs in rows:
        def span(role, f=lambda r: r.t_exit):
            v = [f(r) for r in rs if ROLE[r.role_cta >> 24] == role]
            return (min(v), max(v)) if v else (None, None)
        if kind == "prologue":
            rel = [r.t_release for r in rs if ROLE[r.role_cta >> 24] == "topk" and r.t_release]
            tk_end = span("topk")[1]
            pj = (span("projection", lambda r: r.t_entry)[0], span("projection")[1])
            print("%5d  prologue  topk release %.2f..%.2f end %.2f | projection %s..%s" % (
                lid, us(min(rel)), us(max(rel)), us(tk_end),
                "%.2f" % us(pj[0]) if pj[0] else "-", "%.2f" % us(pj[1]) if pj[1] else "-"))
            layer_phases.append({"release": min(rel), "topk_end": tk_end})
        else:
            a_end = span("attention")[1]
            s_start = span("selection", lambda r: r.t_entry)[0]
            s_end = span("selection")[1]
            print("%5d  attend    selection start %.2f end %.2f | attention end %.2f" % (
                lid, us(s_start), us(s_end), us(a_end)))
            if layer_phases:
                layer_phases[-1].update({"score_start": s_start, "attn_end": a_end, "sel_end": s_end})
    print("\nper layer, us after the prologue's top-k release:")
    print("layer  topk_end  attn_end  sel_end  next_release")
    for i in range(len(layer_phases) - 1):
        p, q = layer_phases[i], layer_phases[i + 1]
        if "attn_end" not in p:
            continue
        r0 = p["release"]
        print("%5d  %8.2f  %8.2f  %7.2f  %12.2f" % (i, (p["topk_end"] - r0) / 1e3, (p["attn_end"] - r0) / 1e3,
                                                 (p["sel_end"] - r0) / 1e3, (q["release"] - r0) / 1e3))


if __name__ == "__main__":
    main()
