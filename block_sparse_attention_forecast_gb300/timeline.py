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

    python -m block_sparse_attention_forecast_gb300.timeline --attn-chain [--layers 32]

instead times the standalone block-sparse decode attention alone, launched once per layer back
to back from a CUDA graph (the step's own selections), and prints per launch its CTAs' phases in
microseconds from the previous launch's last CTA exit (each launch lets the next begin at once,
so CTAs of the next may enter early and wait): entry (first, median), first block in shared
memory (median, max), exit (median, max), and the period (this launch's last exit).
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
    ap.add_argument("--attn-chain", action="store_true",
                    help="time the standalone attention launched back to back, one launch per layer")
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
    if args.attn_chain:
        attn_chain(stack, read, sb, bench, torch)
        return
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



def attn_chain(stack, read, sb, bench, torch):
    """The standalone attention of every layer, back to back in one CUDA graph."""
    stack.advance = False
    stack.run()                                       # every layer's selection
    torch.cuda.synchronize()
    sh, B, n = stack.shape, stack.batch, stack.n_layers

    def loop(s):
        for L in range(n):
            sb.sparda_sparse_decode_attn(sh, stack.layers[L], stack.q[L], stack.idx[L], stack.cnt[L],
                                         stack.seq_len, B, stack.out[L], stack.ws_attn, stream=s)
    t = bench.graph_time(loop, 1)                     # captures and replays once more
    cnt = ctypes.c_int32(0)
    read(None, 0, ctypes.byref(cnt), 1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        loop(torch.cuda.current_stream())
    read(None, 0, ctypes.byref(cnt), 1)               # the capture's own launches record nothing
    g.replay()
    torch.cuda.synchronize()
    cap = 1 << 16
    buf = (Rec * cap)()
    assert read(ctypes.addressof(buf), cap, ctypes.byref(cnt), 1) == 0
    by_launch = {}
    for r in buf[:cnt.value]:
        by_launch.setdefault(r.launch, []).append(r)
    launches = sorted(by_launch)
    print("%d launches, %.2f us per launch (graph replay, CUDA events)" % (n, t / n * 1e6))
    # Each launch lets the next begin at once, so the next one's CTAs may enter (and wait) long
    # before this one ends: phases are measured from the previous launch's last CTA exit (the
    # first launch: from its own first entry).
    print("launch  CTAs  entry first/med  first_block med/max  exit med/max  period"
          "  (us from the previous launch's last exit)")
    prev_end = None
    for lid in launches:
        rs = by_launch[lid]
        t0 = prev_end if prev_end is not None else min(r.t_entry for r in rs)
        ent = np.array([(r.t_entry - t0) / 1e3 for r in rs])
        first = np.array([(r.t_release - t0) / 1e3 for r in rs if r.t_release])
        ex = np.array([(r.t_exit - t0) / 1e3 for r in rs])
        print("%5d  %4d  %6.2f %6.2f  %6.2f %6.2f  %6.2f %6.2f  %6.2f" % (
            lid, len(rs), ent.min(), np.median(ent), np.median(first) if len(first) else -1,
            first.max() if len(first) else -1, np.median(ex), ex.max(), ex.max()))
        prev_end = max(r.t_exit for r in rs)

if __name__ == "__main__":
    main()
