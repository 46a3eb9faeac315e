"""Benchmark of the forecast-driven block-sparse decode step on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload (one "step" = one decode token for every sequence through the whole stack): 32
layers, batch 16, context 131072 tokens, 32 query heads / 2 KV heads / head_dim 128, forecast
projection 4096 -> 256 per layer (layer 0 also has its same-layer head), compression window
32/16, 64-token blocks, top-32 blocks plus block 0 and the tail block, KV resident in HBM
(64 GiB), 16 planted high-score blocks per (layer, sequence, group). Inputs are seeded
synthetic bf16 N(0,1) (weights N(0, 0.02^2)). The K timed steps are consecutive decode
positions ending at context 131072. Prints one JSON line (rank 0).

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

N_LAYERS, BATCH, CTX, G, H, D, HIDDEN, TOPK, PLANTED = 32, 16, 131072, 2, 16, 128, 4096, 32, 16
METRIC = "decode tok/s @128K ctx (B=16 resident, B=64 offload); select+attn HBM GB/s"
def workload_name(n_layers=N_LAYERS):
    return "%d-layer forecast-driven block-sparse decode step, batch 16, context 131072, KV resident" % n_layers


WORKLOAD = workload_name()


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-offload", action="store_true", help="skip the batch-64 offload measurement")
    p.add_argument("--offload-steps", type=int, default=20)
    p.add_argument("--no-selector-ab", action="store_true", help="skip the selector A/B sweep")
    p.add_argument("--no-prefill", action="store_true", help="skip the chunked-prefill A/B")
    p.add_argument("--layout", default="pipelined", choices=["pipelined", "fused"],
                   help="launch layout of the resident step (the same arithmetic in each)")
    p.add_argument("--layers", type=int, default=N_LAYERS,
                   help="layers of the resident stack (the metric is quoted on 32; fewer only for small "
                        "profiler captures)")
    return p.parse_args()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# the sources each profiled kernel is built from (a change to any of them voids its counters)
KERNEL_SOURCES = {
    "attend_and_score": ("fused.cu", "attn_body.cuh", "select_body.cuh", "topk.cuh", "common.cuh", "kernels.h",
                         "timeline.cuh"),
    "attend_and_select": ("fused.cu", "attn_body.cuh", "select_body.cuh", "topk.cuh", "common.cuh", "kernels.h",
                          "timeline.cuh"),
    "decode_prologue": ("prologue.cu", "append_body.cuh", "project_body.cuh", "topk.cuh", "common.cuh",
                        "kernels.h", "timeline.cuh"),
    "sparse_decode_attn": ("attn.cu", "attn_body.cuh", "common.cuh", "kernels.h", "timeline.cuh"),
    "forecast_select": ("select.cu", "select_body.cuh", "topk.cuh", "common.cuh", "kernels.h"),
}


def source_sha(kernel):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "block_sparse_attention_forecast_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """DRAM bytes (read + write) per launch from the committed ncu summary
    (profiles/traffic.json), if the kernel's sources still match the ones profiled; else
    None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            t = json.load(fh)
    except OSError:
        return None
    e = t.get(kernel)
    if not e or e.get("source_sha") != source_sha(kernel):
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), "sparda_clocks_%d_%d.csv" % (os.getpid(), device_index))

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "samples": len(rows),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------- workload
def build_workload(device, seed, steps_total, n_layers=N_LAYERS, layout="pipelined"):
    import torch
    import synth
    import block_sparse_attention_forecast_gb300.binding as sb
    from block_sparse_attention_forecast_gb300.step import DecodeStack

    shape = sb.Shape(n_groups=G, topk=TOPK, max_ctx=CTX, max_batch=BATCH)
    T0 = CTX - steps_total + 1          # the last step runs at context CTX
    nb = CTX // 64
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    W_self0 = synth.normal_bf16_device((G * D, HIDDEN), seed * 1000 + 1, device, std=0.02)
    W_next = [synth.normal_bf16_device((G * D, HIDDEN), seed * 1000 + 2 + L, device, std=0.02)
              for L in range(n_layers - 1)]
    h = synth.normal_bf16_device((n_layers, BATCH, HIDDEN), seed * 1000 + 40, device)
    layers = []
    import numpy as np
    for L in range(n_layers):
        layer = sb.LayerKV.empty(shape, device=device)
        layer.k.copy_(synth.normal_bf16_device(layer.k.shape, seed * 1000 + 100 + L, device))
        layer.v.copy_(synth.normal_bf16_device(layer.v.shape, seed * 1000 + 200 + L, device))
        # planted blocks, shifted along the forecast that selects this layer's blocks
        Wsel, hsel = (W_self0, h[0]) if L == 0 else (W_next[L - 1], h[L - 1])
        direction = (hsel.float() @ Wsel.float().T).view(BATCH, G, D)
        blocks = np.stack([[synth.planted_blocks(seed, (T0 - 1) // 64 + 1, PLANTED, L, b, gg)
                            for gg in range(G)] for b in range(BATCH)])
        synth.plant_batched(layer.k, blocks, direction)
        sb.sparda_compress_keys(shape, layer, torch.full((BATCH,), T0 - 1, dtype=torch.int32, device=device), BATCH)
        layers.append(layer)
    stack = DecodeStack(shape, layers, W_self0, W_next, BATCH, device=device, advance=True, mode=layout)
    stack.h.copy_(h)
    stack.q.copy_(synth.normal_bf16_device(stack.q.shape, seed * 1000 + 41, device))
    stack.k_new.copy_(synth.normal_bf16_device(stack.k_new.shape, seed * 1000 + 42, device))
    stack.v_new.copy_(synth.normal_bf16_device(stack.v_new.shape, seed * 1000 + 43, device))
    stack.seq_len.fill_(T0)
    torch.cuda.synchronize()
    return shape, stack, T0


def kernel_times(stack, reps=4):
    """Average device time of one launch of each hot kernel, from the step's own calls (same
    buffers, every layer) captured back to back in a CUDA graph, replayed and timed with CUDA
    events on the launching stream (no host launch overhead): the step's attend-and-score
    and decode-prologue launches, and for comparison the attend-and-select launch of the
    three-launch layout and forecast_select and sparse_decode_attn each launched alone."""
    import block_sparse_attention_forecast_gb300.binding as sb
    sh, B, n = stack.shape, stack.batch, stack.n_layers
    scores = (stack.ws_sel, stack.ws_sel2)
    # Each attend-and-score / attend-and-select launch lets the next one begin while it runs,
    # so consecutive launches must not share a selection workspace: they alternate by launch
    # count, also across the captured repetitions (31 launches each). Two suffice here: the
    # grid holds one CTA on every SM, so a launch is fully resident, and the one after it can
    # begin, only once the launch before it has exited.
    launch = [0]

    def next_scores():
        launch[0] += 1
        return scores[launch[0] % 2]

    def score_loop(s):
        for L in range(n - 1):
            sb.sparda_attend_and_score(sh, stack.layers[L], stack.q[L], stack.idx[L], stack.cnt[L], stack.out[L],
                                       stack.ws_attn, stack.layers[L + 1].ck, stack.f[L + 1], next_scores(),
                                       stack.seq_len, B, l2_next=stack.W_next[L + 1] if L + 2 < n else None,
                                       stream=s)

    def prologue_loop(s):
        # the prologues of layers 1 .. n-2 (top-k, append and projection each); the scores
        # they select from are the ones score_loop left
        for L in range(1, n - 1):
            sb.sparda_decode_prologue(sh, stack.layers[L], stack.k_new[L], stack.v_new[L], stack.seq_len, B,
                                      ws_scores=scores[L % 2], idx=stack.idx[L], cnt=stack.cnt[L],
                                      W_next=stack.W_next[L], h=stack.h[L], forecast_next=stack.f[L + 1].view(B, -1),
                                      stream=s)

    def fused_loop(s):
        for L in range(n - 1):
            sb.sparda_attend_and_select(sh, stack.layers[L], stack.q[L], stack.idx[L], stack.cnt[L], stack.out[L],
                                        stack.ws_attn, stack.layers[L + 1].ck, stack.f[L + 1], stack.idx[L + 1],
                                        stack.cnt[L + 1], next_scores(), stack.seq_len, B, stream=s)

    def sel_loop(s):
        for L in range(1, n):
            sb.sparda_forecast_select(sh, stack.layers[L].ck, stack.f[L], stack.seq_len, B, stack.idx[L],
                                      stack.cnt[L], stack.ws_sel, stream=s)

    def attn_loop(s):
        for L in range(n):
            sb.sparda_sparse_decode_attn(sh, stack.layers[L], stack.q[L], stack.idx[L], stack.cnt[L],
                                         stack.seq_len, B, stack.out[L], stack.ws_attn, stream=s)

    out = {}
    for name, fn, per in (("score", score_loop, n - 1), ("prologue", prologue_loop, n - 2),
                          ("fused", fused_loop, n - 1), ("select", sel_loop, n - 1), ("attn", attn_loop, n)):
        if per > 0:
            out[name] = graph_time(fn, reps) / per
    return out


def select_bytes(T, batch=BATCH):
    """Algorithmic bytes of one selection launch: every compressed key of the windows complete
    within T-1 tokens plus the forecast, per (sequence, group)."""
    from block_sparse_attention_forecast_gb300.binding import num_windows
    return batch * G * (num_windows(T - 1) * D * 2 + D * 2)


def attn_bytes(batch=BATCH):
    """Algorithmic bytes of one attention launch: K and V of the k + 2 selected 64-token blocks
    plus the 16 queries read and the 16 outputs written, per (sequence, group)."""
    return batch * G * ((TOPK + 2) * 64 * D * 2 * 2 + 2 * H * D * 2)


def prologue_bytes(batch=BATCH, topk=True):
    """Algorithmic bytes of one decode prologue: the forecast head's weights and the hidden
    states read and the forecasts written (projection), the block scores read and the
    selection written (top-k, if it runs there), the token's key and value read and written
    (append)."""
    nb = CTX // 64
    proj = G * D * HIDDEN * 2 + batch * HIDDEN * 2 + batch * G * D * 2
    sel = batch * G * (nb * 4 + (TOPK + 2) * 4 + 4) if topk else 0
    append = batch * G * D * 2 * 2 * 2
    return proj + sel + append


def replica_max(values, dist, device):
    """Max over ranks of each timing (every rank gets the maxima). With one rank the values
    come back unchanged."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def replica_throughput(world, batch, steps, elapsed_max):
    """Whole-job decode tokens/s of `world` independent replicas, each decoding `batch`
    sequences for `steps` steps, timed by the slowest replica."""
    return world * batch * steps / elapsed_max


# ---------------------------------------------------------------------- host placement
def gpu_pci_dir(device_index):
    """sysfs directory of the GPU's PCI function, from nvidia-smi's bus id (None if unknown)."""
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(device_index), "--query-gpu=pci.bus_id",
                              "--format=csv,noheader"], capture_output=True, text=True, timeout=30).stdout.strip()
    except (OSError, subprocess.TimeoutExpired):
        return None
    if not out:
        return None
    dom, rest = out.split(":", 1)
    path = "/sys/bus/pci/devices/%s:%s" % (dom[-4:].lower(), rest.lower())
    return path if os.path.isdir(path) else None


def parse_cpulist(text):
    cpus = set()
    for part in text.strip().split(","):
        if not part:
            continue
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        else:
            cpus.add(int(part))
    return cpus


def numa_nodes_of(addr):
    """{node: pages} of the mapping holding address `addr`, from /proc/self/numa_maps."""
    try:
        with open("/proc/self/maps") as fh:
            start = None
            for line in fh:
                lo, hi = (int(x, 16) for x in line.split()[0].split("-"))
                if lo <= addr < hi:
                    start = lo
                    break
        if start is None:
            return None
        with open("/proc/self/numa_maps") as fh:
            for line in fh:
                f = line.split()
                if int(f[0], 16) == start:
                    return {k[1:]: int(v) for k, v in (x.split("=") for x in f[1:] if x.startswith("N") and "=" in x)}
    except (OSError, ValueError):
        return None
    return None


def host_placement(device_index):
    """The GPU's PCI NUMA node and its local CPUs (from sysfs); None where unknown."""
    d = gpu_pci_dir(device_index)
    info = {"gpu_pci": d, "gpu_numa_node": None, "gpu_local_cpus": None}
    if d:
        try:
            with open(os.path.join(d, "numa_node")) as fh:
                info["gpu_numa_node"] = int(fh.read().strip())
            with open(os.path.join(d, "local_cpulist")) as fh:
                info["gpu_local_cpus"] = sorted(parse_cpulist(fh.read()))
        except (OSError, ValueError):
            pass
    return info


# ---------------------------------------------------------------------- offloaded decode
OFF_BATCH, OFF_DISTINCT, OFF_FFN = 64, 4, 14336


def graph_time(fn, reps=1):
    """Device time of `reps` captured repetitions of fn(stream), per repetition (seconds)."""
    import torch
    s = torch.cuda.current_stream()
    fn(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        for _ in range(reps):
            fn(cs)
    g.replay()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    g.replay()
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e-3 / reps


def pinned_h2d_gbs(device, nbytes=1 << 30):
    """Host-to-device bandwidth of one copy from a pinned buffer (allocated here, by the calling
    thread) to device memory, best of 3 (GB/s)."""
    import torch
    hb = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    hb.fill_(1)
    db = torch.empty(nbytes, dtype=torch.uint8, device=device)
    db.copy_(hb)
    torch.cuda.synchronize()
    best = 0.0
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        db.copy_(hb, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del hb, db
    return best


def run_offload(device, seed, steps, warmup):
    """The offloaded decode step: batch 64, context 131072, 32 layers; layer 0 resident, layers
    1-31 with their K/V in pinned host memory (gathered over the host link by the persistent
    UVA kernel on a side stream), compressed keys and hot blocks in HBM, and a stand-in bf16
    FFN GEMM [64 x 4096] x [4096 x 14336] after every attention. 31 layers of K/V at this size
    would take ~266 GB of pinned host memory, more than a host with a few hundred GB can pin
    beside everything else, so the host holds 4 distinct K/V pairs (8.6 GB each) shared
    round-robin by layers 1-31; aliasing leaves the bytes gathered per step unchanged. Measured with the gather
    overlapped, with it waited on right after selection, and against the same step with
    every layer resident (4 distinct resident K/V pairs, same aliasing)."""
    import gc
    import torch
    import synth
    import block_sparse_attention_forecast_gb300.binding as sb
    from block_sparse_attention_forecast_gb300.step import DecodeStack
    B = OFF_BATCH
    shape = sb.Shape(n_groups=G, topk=TOPK, max_ctx=CTX, max_batch=B)
    # the pinned host pool on the memory nearest the GPU: this thread runs on the GPU's local
    # CPUs while it allocates and first touches the pool (the default local-allocation policy)
    placement = host_placement(torch.cuda.current_device())
    link_before_binding = pinned_h2d_gbs(device)
    affinity = os.sched_getaffinity(0)
    local = set(placement["gpu_local_cpus"] or []) & affinity
    if local:
        os.sched_setaffinity(0, local)
    steps_total = 1 + warmup + steps
    T0 = CTX - steps_total + 1
    seq_c = torch.full((B,), T0 - 1, dtype=torch.int32, device=device)
    devK, devV, hostK, hostV, cks = [], [], [], [], []
    for i in range(OFF_DISTINCT):
        kd = synth.normal_bf16_device((B, G, CTX, D), seed * 1000 + 500 + i, device)
        vd = synth.normal_bf16_device((B, G, CTX, D), seed * 1000 + 600 + i, device)
        ck = torch.zeros((B, G, shape.w_cap, D), dtype=torch.bfloat16, device=device)
        sb.sparda_compress_keys(shape, sb.LayerKV(kd, vd, ck), seq_c, B)
        hk = torch.empty(kd.shape, dtype=torch.bfloat16, pin_memory=True)
        hv = torch.empty(vd.shape, dtype=torch.bfloat16, pin_memory=True)
        hk.copy_(kd)
        hv.copy_(vd)
        devK.append(kd); devV.append(vd); hostK.append(hk); hostV.append(hv); cks.append(ck)
    layers = [sb.LayerKV(devK[0], devV[0], cks[0].clone())]
    for L in range(1, N_LAYERS):
        i = (L - 1) % OFF_DISTINCT
        layer = sb.LayerKV(hostK[i], hostV[i], cks[i].clone(),
                           torch.zeros((B, G, 3, 64, D), dtype=torch.bfloat16, device=device),
                           torch.zeros((B, G, 3, 64, D), dtype=torch.bfloat16, device=device), True)
        sb.fill_hot_from_host(layer, [T0 - 1] * B)
        layers.append(layer)
    resident = [layers[0]] + [sb.LayerKV(devK[(L - 1) % OFF_DISTINCT], devV[(L - 1) % OFF_DISTINCT], layers[L].ck)
                              for L in range(1, N_LAYERS)]
    W_self0 = synth.normal_bf16_device((G * D, HIDDEN), seed * 1000 + 701, device, std=0.02)
    W_next = [synth.normal_bf16_device((G * D, HIDDEN), seed * 1000 + 702 + L, device, std=0.02)
              for L in range(N_LAYERS - 1)]
    Wffn = [synth.normal_bf16_device((HIDDEN, OFF_FFN), seed * 1000 + 800 + i, device, std=0.02)
            for i in range(OFF_DISTINCT)]
    x = synth.normal_bf16_device((B, HIDDEN), seed * 1000 + 810, device)
    y = torch.empty((B, OFF_FFN), dtype=torch.bfloat16, device=device)

    def ffn(L):
        torch.mm(x, Wffn[L % OFF_DISTINCT], out=y)

    def make(lays, overlap, block_cache=None):
        st = DecodeStack(shape, lays, W_self0, W_next, B, device=device, overlap=overlap, advance=True,
                         after_attention=ffn, block_cache=block_cache)
        st.h.copy_(synth.normal_bf16_device(st.h.shape, seed * 1000 + 820, device))
        st.q.copy_(synth.normal_bf16_device(st.q.shape, seed * 1000 + 821, device))
        st.k_new.copy_(synth.normal_bf16_device(st.k_new.shape, seed * 1000 + 822, device))
        st.v_new.copy_(synth.normal_bf16_device(st.v_new.shape, seed * 1000 + 823, device))
        return st

    def time_stack(st, h_bank=None):
        """Mean step time; with h_bank, every step first takes the next hidden states of the bank
        (a device copy on the same stream), so that consecutive steps select different blocks."""
        st.seq_len.fill_(T0)
        st.capture()
        for i in range(warmup):
            if h_bank is not None:
                st.h.copy_(h_bank[i % len(h_bank)])
            st.run()
        torch.cuda.synchronize()
        if st.cache_stats is not None:
            st.cache_stats.zero_()
        s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for i in range(steps):
            if h_bank is not None:
                st.h.copy_(h_bank[(warmup + i) % len(h_bank)])
            st.run()
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e-3 / steps

    res = {}
    st_ov = make(layers, True)
    t_ov = time_stack(st_ov)
    st_pg = make(layers, True)
    st_pg.gather_ctas = 32                  # the pages' H100 setting for batch >= 32, for context
    t_pages = time_stack(st_pg)
    del st_pg
    t_no = time_stack(make(layers, False))
    t_res = time_stack(make(resident, True))
    # the cross-step block cache (an extension beyond the pages): each offloaded layer keeps
    # topk + 2 gathered blocks per (sequence, group) in HBM and gathers only the ones it lacks.
    # Measured with the hidden states constant across steps (consecutive steps select nearly
    # the same blocks: the best case) and with new hidden states every step (independent
    # selections: the worst case); real decoding lies between.
    cache_res = {}
    h_bank = [synth.normal_bf16_device((N_LAYERS, B, HIDDEN), seed * 1000 + 830 + i, device) for i in range(4)]
    for name, bank in (("same_hidden_every_step", None), ("new_hidden_every_step", h_bank)):
        st_bc = make(layers, True, block_cache=TOPK + 2)
        t_bc = time_stack(st_bc, bank)
        hits, misses = st_bc.cache_stats.cpu().tolist()
        cache_res[name] = {"tok_s": B / t_bc, "ms_per_step": t_bc * 1e3, "hit_rate": hits / max(1, hits + misses),
                           "blocks_gathered_per_step": misses / steps,
                           "offload_vs_resident_time": t_bc / t_res}
        del st_bc
        gc.collect()
        torch.cuda.empty_cache()
    del h_bank
    # between the two: hidden states that drift from step to step, h <- sqrt(1 - eps^2) h + eps z
    # with fresh noise z, from the stack's own starting states (so the planted blocks stay
    # relevant), which keeps part of consecutive steps' selections
    for eps in (0.05, 0.2):
        st_bc = make(layers, True, block_cache=TOPK + 2)
        walk, h = [], st_bc.h.float()
        for i in range(warmup + steps):
            z = synth.normal_bf16_device(st_bc.h.shape, seed * 1000 + 840 + i, device).float()
            h = (1.0 - eps * eps) ** 0.5 * h + eps * z
            walk.append(h.to(torch.bfloat16))
        t_bc = time_stack(st_bc, walk)
        hits, misses = st_bc.cache_stats.cpu().tolist()
        cache_res["hidden_drift_%g" % eps] = {"tok_s": B / t_bc, "ms_per_step": t_bc * 1e3,
                                              "hit_rate": hits / max(1, hits + misses),
                                              "blocks_gathered_per_step": misses / steps,
                                              "offload_vs_resident_time": t_bc / t_res}
        del st_bc, walk, h
        gc.collect()
        torch.cuda.empty_cache()
    cache_res["slots_per_group"] = TOPK + 2
    # without the cache, at new hidden states every step (the comparison for the worst case)
    h_bank = [synth.normal_bf16_device((N_LAYERS, B, HIDDEN), seed * 1000 + 830 + i, device) for i in range(4)]
    st_nb = make(layers, True)
    cache_res["no_cache_new_hidden_every_step_tok_s"] = B / time_stack(st_nb, h_bank)
    del st_nb, h_bank
    gc.collect()
    torch.cuda.empty_cache()
    # the gather alone: the step's own 31 gathers (last step's selections), per launch
    gbytes = B * G * TOPK * 2 * 64 * D * 2

    def gathers(n_ctas):
        def fn(s):
            for L in range(1, N_LAYERS):
                sb.sparda_prefetch_blocks(shape, st_ov.layers[L], st_ov.idx[L], st_ov.cnt[L], st_ov.seq_len, B,
                                          st_ov.stage_k[L % 2], st_ov.stage_v[L % 2], n_ctas, stream=s)
        return graph_time(fn) / (N_LAYERS - 1)
    st_ov.seq_len.fill_(CTX)
    sweep = {}
    for n in (8, 16, 32, 64, 152):
        sweep[str(n)] = gbytes / gathers(n) / 1e9
    t_g = gathers(0)
    # the copy-engine alternative for one layer's gather: the selection read back to the host,
    # then one cudaMemcpyAsync per run of consecutive selected blocks (K and V); wall time from
    # the selection on the device to the copies done, and the copies' own device time
    L1 = 1
    ce_times, ce_dev, n_copies = [], [], 0
    for rep in range(3):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ih, ch, sh = st_ov.idx[L1].cpu(), st_ov.cnt[L1].cpu(), st_ov.seq_len.cpu()     # each waits on the device
        s_ce = torch.cuda.current_stream()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(s_ce)
        n_copies = sb.sparda_prefetch_blocks_copy_engine(shape, st_ov.layers[L1], ih, ch, sh, B, st_ov.stage_k[0],
                                                         st_ov.stage_v[0], stream=s_ce)
        a1.record(s_ce)
        torch.cuda.synchronize()
        ce_times.append(time.perf_counter() - t0)
        ce_dev.append(a0.elapsed_time(a1) * 1e-3)
    ce = {"copies_per_layer": n_copies, "wall_ms_per_layer": min(ce_times) * 1e3,
          "device_ms_per_layer": min(ce_dev) * 1e3, "gbs_wall": gbytes / min(ce_times) / 1e9,
          "vs_sm_gather_time": min(ce_times) / t_g}
    h2d = pinned_h2d_gbs(device)              # pinned on the GPU-local node (bound above)
    placement["pool_numa_pages"] = numa_nodes_of(hostK[0].data_ptr())
    placement["bound_to_local_cpus"] = bool(local)
    placement["h2d_gbs_before_binding"] = link_before_binding
    placement["h2d_gbs_local"] = h2d
    os.sched_setaffinity(0, affinity)
    link = max([h2d, link_before_binding] + list(sweep.values()))
    res.update({
        "workload": "32-layer decode step, batch 64, context 131072, layers 1-31 K/V in pinned host memory, "
                    "stand-in FFN GEMM 64x4096x14336 per layer",
        "tok_s_overlap": B / t_ov, "tok_s_no_overlap": B / t_no, "tok_s_resident_same_shapes": B / t_res,
        "ms_per_step_overlap": t_ov * 1e3, "ms_per_step_no_overlap": t_no * 1e3,
        "ms_per_step_resident": t_res * 1e3, "offload_vs_resident_time": t_ov / t_res,
        "tok_s_overlap_32_copy_ctas": B / t_pages,
        "gather_us_per_layer": t_g * 1e6, "gather_bytes_per_layer": gbytes,
        "gather_gbs": gbytes / t_g / 1e9, "gather_cta_default": sb.sparda_prefetch_default_ctas(B),
        "gather_cta_sweep_gbs": sweep, "link_h2d_copy_gbs": h2d,
        "gather_link_frac": (gbytes / t_g / 1e9) / link,
        "gather_gbs_while_overlapping": (N_LAYERS - 1) * gbytes / t_ov / 1e9,
        "gather_link_frac_while_overlapping": (N_LAYERS - 1) * gbytes / t_ov / 1e9 / link,
        "link_peak_gbs": link,
        "host_buffers": "4 distinct 8.6 GB K/V pairs aliased over layers 1-31 (bytes gathered per step unchanged)",
        "block_cache": cache_res,
        "host_placement": placement,
        "copy_engine_gather": ce,
        "device_error_flags": sb.sparda_device_error(clear=True),
    })
    del st_ov, layers, resident, devK, devV, hostK, hostV, cks
    gc.collect()
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------- selector A/B
def selector_ab(device, seed):
    """The selector A/B: one layer's selection, the Forecast selector (one head per group, no
    softmax) against the baseline multi-head selector (16 query heads per group, softmax per
    head, sum, max-pool, top-32), for batch 1..128 at context 131072 and for context 32K..128K
    at batch 16. Compressed keys, forecasts and queries are seeded N(0,1) bf16 drawn on the
    device (selection time does not depend on their values). Device time per call from CUDA
    graph replays; GB/s counts every byte each call moves (compressed keys, forecast or
    queries, block scores written and read back, selection)."""
    import torch
    import synth
    import block_sparse_attention_forecast_gb300.binding as sb
    out = {"batch_sweep_ctx131072": {}, "context_sweep_batch16": {}}

    def one(B, T):
        shape = sb.Shape(n_groups=G, topk=TOPK, max_ctx=T, max_batch=B)
        ck = synth.normal_bf16_device((B, G, shape.w_cap, D), seed * 1000 + 900 + B, device, std=0.18)
        f = synth.normal_bf16_device((B, G, D), seed * 1000 + 901, device)
        q = synth.normal_bf16_device((B, G * H, D), seed * 1000 + 902, device)
        seq = torch.full((B,), T, dtype=torch.int32, device=device)
        idx = torch.zeros((B, G, TOPK + 2), dtype=torch.int32, device=device)
        cnt = torch.zeros((B, G), dtype=torch.int32, device=device)
        ws = sb.workspace(shape, B, sb.WS_SELECT, device)
        wm = sb.workspace(shape, B, sb.WS_MULTIHEAD, device)
        from block_sparse_attention_forecast_gb300.binding import num_windows
        W = num_windows(T - 1)
        t_f = graph_time(lambda s: sb.sparda_forecast_select(shape, ck, f, seq, B, idx, cnt, ws, stream=s), 8)
        t_m = graph_time(lambda s: sb.sparda_multihead_select(shape, ck, q, seq, B, idx, cnt, wm, stream=s), 8)
        # every byte each call moves: the compressed keys, the forecast (or the 16 queries), the
        # float32 block scores written and read back by the top-k, and the selection written
        nb = (T - 1) // 64 + 1
        tail = nb * 4 * 2 + (TOPK + 2) * 4 + 4
        bytes_f = B * G * (W * D * 2 + D * 2 + tail)
        bytes_m = B * G * (W * D * 2 + H * D * 2 + tail)
        del ck, ws, wm
        torch.cuda.empty_cache()
        return {"forecast_us": t_f * 1e6, "multihead_us": t_m * 1e6, "speedup": t_m / t_f,
                "forecast_gbs": bytes_f / t_f / 1e9, "multihead_gbs": bytes_m / t_m / 1e9}

    for B in (1, 8, 32, 64, 128):
        out["batch_sweep_ctx131072"][str(B)] = one(B, CTX)
    for T in (32768, 65536, 98304, 131072):
        out["context_sweep_batch16"][str(T)] = one(16, T)
    out["device_error_flags"] = sb.sparda_device_error(clear=True)
    return out


# ---------------------------------------------------------------------- chunked prefill A/B
def prefill_attn_flops(idx, cnt, T):
    """Algorithmic flops of the causal block-sparse prefill attention of one sequence-group:
    QK^T and PV (2 x 2 flops per query head, key and dimension) over the keys each token
    attends, from the chunk selections idx [n_chunks, k+2] / cnt [n_chunks] on the host."""
    keys = 0
    for c in range((T + 63) // 64):
        n_tok = min(64, T - 64 * c)
        full = int(cnt[c]) - 1                           # selected blocks before the chunk's own
        keys += n_tok * 64 * full + n_tok * (n_tok + 1) // 2
    return keys * H * D * 4


def prefill_ab(device, seed, contexts=(32768, 65536, 131072)):
    """One layer's prefill of a batch-1 prompt at each context: the Forecast chunk selector
    against the baseline multi-head chunk selector, and the causal block-sparse prefill
    attention over the forecast's selections (top-32 blocks plus block 0 and the chunk's own).
    K, V, queries and per-token forecasts are seeded N(0,1) bf16 drawn on the device. Device
    time per call from CUDA graph replays."""
    import torch
    import synth
    import block_sparse_attention_forecast_gb300.binding as sb
    peaks, _ = measured_peaks()
    out = {}
    for T in contexts:
        shape = sb.Shape(n_groups=G, topk=TOPK, max_ctx=T, max_batch=1)
        layer = sb.LayerKV.empty(shape, device=device)
        layer.k.copy_(synth.normal_bf16_device(layer.k.shape, seed * 1000 + 950, device))
        layer.v.copy_(synth.normal_bf16_device(layer.v.shape, seed * 1000 + 951, device))
        q = synth.normal_bf16_device((1, T, G * H, D), seed * 1000 + 952, device)
        f = synth.normal_bf16_device((1, T, G, D), seed * 1000 + 953, device)
        seq = torch.full((1,), T, dtype=torch.int32, device=device)
        sb.sparda_compress_keys(shape, layer, seq, 1)
        nc = T // 64
        idx = torch.zeros((1, G, nc, TOPK + 2), dtype=torch.int32, device=device)
        cnt = torch.zeros((1, G, nc), dtype=torch.int32, device=device)
        idx_m, cnt_m = torch.zeros_like(idx), torch.zeros_like(cnt)
        ws = sb.workspace(shape, 1, sb.WS_PREFILL, device)
        o = torch.empty_like(q)
        t_f = graph_time(lambda s: sb.sparda_prefill_forecast_select(shape, layer.ck, f, seq, 1, idx, cnt, ws,
                                                                     stream=s), 3)
        t_m = graph_time(lambda s: sb.sparda_prefill_multihead_select(shape, layer.ck, q, seq, 1, idx_m, cnt_m, ws,
                                                                      stream=s), 1)
        t_a = graph_time(lambda s: sb.sparda_prefill_attn(shape, layer, q, idx, cnt, seq, 1, o, stream=s), 2)
        ic, cc = idx.cpu().numpy(), cnt.cpu().numpy()
        flops = sum(prefill_attn_flops(ic[0, g], cc[0, g], T) for g in range(G))
        tf = flops / t_a / 1e12
        out[str(T)] = {
            "forecast_select_ms": t_f * 1e3, "multihead_select_ms": t_m * 1e3, "attn_ms": t_a * 1e3,
            "selection_speedup": t_m / t_f,
            "prefill_tok_s_forecast": T / (t_f + t_a), "prefill_tok_s_multihead": T / (t_m + t_a),
            "prefill_speedup": (t_m + t_a) / (t_f + t_a),
            "attn_tflops": tf, "attn_flops": flops, "attn_frac_of_bf16_peak": tf / float(peaks["bf16_tflops"]),
        }
        del layer, q, f, o, ws, idx, cnt, idx_m, cnt_m
        torch.cuda.empty_cache()
    out["device_error_flags"] = sb.sparda_device_error(clear=True)
    out["workload"] = ("one 8B-shaped layer's prefill, batch 1, 64-token query chunks, top-32 blocks plus block 0 "
                       "and the chunk's own; K/V/queries/forecasts seeded N(0,1) bf16")
    return out


# ---------------------------------------------------------------------- single-kernel cases
def kernel_case(name, batch=16, ctx=CTX, reps=48, seed=0):
    """One kernel alone on a seeded case, for profilers and quick timing: 'attn' (the
    standalone block-sparse decode attention over a forecast selection), 'select' (the
    standalone Forecast selector), 'multihead' (the baseline selector) or 'prefill' (one layer's
    prefill A/B, batch 1). Consecutive launches cycle through input sets whose bytes together
    exceed twice the L2 (different selections for 'attn', different compressed-key buffers for
    the selectors), so no launch finds its data in L2. Prints the mean device time of `reps`
    launches captured back to back in a CUDA graph and the median of single launches after
    an L2 flush (launch latency included), with the algorithmic GB/s."""
    import math
    import torch
    import synth
    import block_sparse_attention_forecast_gb300.binding as sb
    device = "cuda:0"
    if name == "prefill":
        print(json.dumps(prefill_ab(device, seed, (ctx,))))
        return
    B = batch
    l2 = 129 << 20
    shape = sb.Shape(n_groups=G, topk=TOPK, max_ctx=ctx, max_batch=B)
    layer = sb.LayerKV.empty(shape, device=device)
    layer.k.copy_(synth.normal_bf16_device(layer.k.shape, seed * 1000 + 11, device))
    layer.v.copy_(synth.normal_bf16_device(layer.v.shape, seed * 1000 + 12, device))
    seq = torch.full((B,), ctx, dtype=torch.int32, device=device)
    sb.sparda_compress_keys(shape, layer, seq - 1, B)
    q = synth.normal_bf16_device((B, G * H, D), seed * 1000 + 14, device)
    ws = sb.workspace(shape, B, sb.WS_SELECT, device)
    wa = sb.workspace(shape, B, sb.WS_ATTN, device)
    wm = sb.workspace(shape, B, sb.WS_MULTIHEAD, device)
    out = torch.zeros((B, G * H, D), dtype=torch.bfloat16, device=device)
    from block_sparse_attention_forecast_gb300.binding import num_windows
    sel_b = B * G * (num_windows(ctx - 1) * D * 2 + D * 2)
    nbytes = {"attn": attn_bytes(B), "select": sel_b, "multihead": sel_b - B * G * D * 2 + B * G * H * D * 2}[name]
    n_sets = max(1, math.ceil(2 * l2 / nbytes))
    fs = [synth.normal_bf16_device((B, G, D), seed * 1000 + 20 + i, device) for i in range(n_sets)]
    idxs = [torch.zeros((B, G, TOPK + 2), dtype=torch.int32, device=device) for _ in range(n_sets)]
    cnts = [torch.zeros((B, G), dtype=torch.int32, device=device) for _ in range(n_sets)]
    cks = [layer.ck] + [layer.ck.clone() for _ in range(n_sets - 1)] if name != "attn" else [layer.ck]
    for i in range(n_sets):
        sb.sparda_forecast_select(shape, layer.ck, fs[i], seq, B, idxs[i], cnts[i], ws)

    def call(i, s):
        k = i % n_sets
        if name == "attn":
            sb.sparda_sparse_decode_attn(shape, layer, q, idxs[k], cnts[k], seq, B, out, wa, stream=s)
        elif name == "select":
            sb.sparda_forecast_select(shape, cks[k], fs[k], seq, B, idxs[k], cnts[k], ws, stream=s)
        else:
            sb.sparda_multihead_select(shape, cks[k], q, seq, B, idxs[k], cnts[k], wm, stream=s)
    t_chain = graph_time(lambda s: [call(i, s) for i in range(reps)]) / reps
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    st = torch.cuda.current_stream()
    single = []
    for i in range(20):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        call(i, st)
        b.record(st)
        torch.cuda.synchronize()
        single.append(a.elapsed_time(b) * 1e-3)
    single.sort()
    t1 = single[len(single) // 2]
    print(json.dumps({"case": name, "batch": B, "context": ctx, "alg_bytes": nbytes, "input_sets": n_sets,
                      "us_back_to_back": t_chain * 1e6, "gbs_back_to_back": nbytes / t_chain / 1e9,
                      "us_single_after_l2_flush": t1 * 1e6, "gbs_single": nbytes / t1 / 1e9,
                      "device_error_flags": sb.sparda_device_error(clear=True)}))


# ---------------------------------------------------------------------- CPU oracle sample
CPU_SAMPLE_SCRIPT = r"""
import sys, time, json
sys.path.insert(0, %(root)r)
import numpy as np
import synth
from oracle import sparda_oracle as O
units, T = %(units)d, %(T)d
t_total = 0.0
for u in range(units):
    K = synth.normal_bf16((T, 128), 900, u, 1).double().numpy()
    V = synth.normal_bf16((T, 128), 900, u, 2).double().numpy()
    q = synth.normal_bf16((16, 128), 900, u, 3).double().numpy()
    W = synth.normal_bf16((128, 4096), 900, u, 4, std=0.02).double().numpy()
    h = synth.normal_bf16((4096,), 900, u, 5).double().numpy()
    t0 = time.perf_counter()
    f = O.forecast_project(W, h)
    sel = O.forecast_select_one(K, f, T, 32)
    o = O.block_sparse_attention(q, K, V, sel, T)
    t_total += time.perf_counter() - t0
print(json.dumps({"seconds": t_total, "units": units}))
"""


def cpu_oracle_sample(units):
    """Times the oracle on `units` (layer, sequence, group) pieces of the 128K step in a
    single-threaded subprocess; returns (seconds per full step, cores, description)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = CPU_SAMPLE_SCRIPT % {"root": ROOT, "units": units, "T": CTX}
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed: " + r.stderr[-2000:])
    res = json.loads(r.stdout.strip().splitlines()[-1])
    per_unit = res["seconds"] / res["units"]
    per_step = per_unit * N_LAYERS * BATCH * G
    desc = ("%d (layer, sequence, group) units of the 128K step (forecast projection + compressed "
            "keys + select + 16-head attention each), %.2f s per unit, x%d units per step" %
            (units, per_unit, N_LAYERS * BATCH * G))
    return per_step, 1, desc


def _oracle_inputs(u, T=CTX):
    import synth
    return (synth.normal_bf16((T, 128), 900, u, 1).double().numpy(),
            synth.normal_bf16((T, 128), 900, u, 2).double().numpy(),
            synth.normal_bf16((16, 128), 900, u, 3).double().numpy(),
            synth.normal_bf16((128, 4096), 900, u, 4, std=0.02).double().numpy(),
            synth.normal_bf16((4096,), 900, u, 5).double().numpy())


def _oracle_worker(first_unit, n_units, barrier, results, T=CTX):
    """One spawned worker of the all-core oracle baseline: draws its units' inputs, waits for
    every worker, then runs the oracle on them (forecast projection, compressed keys,
    selection, 16-head attention per unit) and reports its start and end times (the monotonic
    clock is shared by the processes of a host)."""
    from oracle import sparda_oracle as O
    inputs = [_oracle_inputs(first_unit + i, T) for i in range(n_units)]
    barrier.wait()
    t0 = time.perf_counter()
    for K, V, q, W, h in inputs:
        f = O.forecast_project(W, h)
        sel = O.forecast_select_one(K, f, T, 32)
        O.block_sparse_attention(q, K, V, sel, T)
    results.put((t0, time.perf_counter()))


def cpu_oracle_parallel(units_per_core=2):
    """The oracle on every core this process may use (os.sched_getaffinity): one
    single-threaded worker process per core (spawned), each on its own (layer, sequence,
    group) units of the 128K step, started together; the wall time from the first start to the
    last end. Returns (seconds per full step, cores, description)."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0))
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    ctx = mp.get_context("spawn")
    barrier, results = ctx.Barrier(cores), ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(1000 + r * units_per_core, units_per_core, barrier, results))
             for r in range(cores)]
    for p in procs:
        p.start()
    spans = [results.get(timeout=1800) for _ in procs]
    for p in procs:
        p.join()
    wall = max(b for _, b in spans) - min(a for a, _ in spans)
    units = units_per_core * cores
    per_step = wall / units * N_LAYERS * BATCH * G
    desc = ("%d (layer, sequence, group) units of the 128K step on %d worker processes (one per core, started "
            "together), %.1f s wall, x%d units per step" % (units, cores, wall, N_LAYERS * BATCH * G))
    return per_step, cores, desc


def run_reference(args):
    """The oracle arm: each step is one (layer, sequence, group) unit of the 128K workload
    (the oracle is far too slow for a whole step); the per-step figure is extrapolated to
    the 1024 units of a full step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    units = max(1, min(args.steps, 40))
    per_step, cores, desc = cpu_oracle_sample(units)
    value = BATCH / per_step
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": units, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch": BATCH, "context": CTX, "layers": N_LAYERS, "topk": TOPK},
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            # each "step" here is one sampled unit; ms_per_step is extrapolated to the 1024 units
            # of a full step, so steps x ms_per_step is far longer than this run takes
            "extrapolated": {"units_timed": units, "units_per_step": N_LAYERS * BATCH * G}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------- main arm
def run_ours(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = "cuda:%d" % local

    cpu = cpu_all = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(24)          # before any heavy GPU setup; ~15 s of CPU work
        cpu_all = cpu_oracle_parallel(3)     # every core, spawned workers; a few seconds

    steps_total = 1 + args.warmup + args.steps
    shape, stack, T0 = build_workload(device, args.seed + rank, steps_total, args.layers, args.layout)
    import block_sparse_attention_forecast_gb300.binding as sb
    stack.capture()                          # one eager step, then the captured graph
    for _ in range(args.warmup):
        stack.run()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")
    e0.record(s)
    for _ in range(args.steps):
        stack.run()
    e1.record(s)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    dev_err = sb.sparda_device_error(clear=True)
    elapsed = e0.elapsed_time(e1) * 1e-3
    T_last = int(stack.seq_len[0].item()) - 1      # context of the last timed step

    # the per-launch kernel times (roofline) before the end-to-end leg, so that its host
    # traffic cannot colour them
    stack.seq_len.fill_(CTX)                 # the kernels below run at context CTX
    kt = kernel_times(stack)
    dev_err |= sb.sparda_device_error(clear=True)

    # end to end through the public API: every step copies its inputs from pinned host memory
    # and its attention outputs back to pinned host memory (DecodeStack.attach_host_io: inside
    # the captured step, the first layers' inputs and the last layers' outputs go by copy
    # kernel on the compute stream, the rest by DMA on the I/O stream, overlapped with the
    # compute); wall-clock time around the replays, synchronised at the end
    host_in = stack.pinned_inputs()
    for n in stack.IO_INPUTS:
        host_in[n].copy_(getattr(stack, n).cpu())
    host_out = torch.zeros_like(stack.out, device="cpu").pin_memory()
    stack.attach_host_io(host_in, host_out)
    h2d, d2h = stack.io_bytes()
    e2e_steps = min(args.steps, 200)
    stack.seq_len.fill_(CTX - e2e_steps - 2)   # the capture's eager step and one replay advance it
    stack.capture()
    stack.run()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        stack.run()
    torch.cuda.synchronize()
    e2e_elapsed = time.perf_counter() - t0
    stack.attach_host_io(None, None)

    launches_per_step = stack.kernel_launches_per_step()
    offload = None
    if world == 1 and not args.no_offload:
        import gc
        del stack
        gc.collect()
        torch.cuda.empty_cache()
        offload = run_offload(device, args.seed, args.offload_steps, 3)
    ab = None
    if world == 1 and not args.no_selector_ab:
        ab = selector_ab(device, args.seed)
    pf = None
    if world == 1 and not args.no_prefill:
        pf = prefill_ab(device, args.seed)
    elapsed, e2e_elapsed = replica_max([elapsed, e2e_elapsed], dist, device)
    if rank != 0:
        dist.destroy_process_group()
        return

    peaks, peak_src = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    sel_b, att_b = select_bytes(CTX), attn_bytes()
    kernels = {}
    for name, key, b in (("attend_and_score", "score", sel_b + att_b), ("attend_and_select", "fused", sel_b + att_b),
                         ("forecast_select", "select", sel_b), ("sparse_decode_attn", "attn", att_b),
                         ("decode_prologue", "prologue", prologue_bytes())):
        if key in kt:
            gbs = b / kt[key] / 1e9
            kernels[name] = {"us": kt[key] * 1e6, "alg_bytes": b, "gbs": gbs, "frac": gbs / hbm}
    # the step's dominant kernel: layer L's attention beside layer L+1's selection
    dom = {"pipelined": "attend_and_score", "fused": "attend_and_select"}[args.layout]
    dk = kernels[dom]
    ms = elapsed / args.steps * 1e3
    value = replica_throughput(world, BATCH, args.steps, elapsed)
    n = args.layers
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name(n), "batch_per_gpu": BATCH, "context": CTX, "layers": n,
                   "layout": args.layout,
                   "kv_heads": G, "q_heads": G * H, "head_dim": D, "topk": TOPK, "block": 64,
                   "window": "32/16", "hidden": HIDDEN, "parallelism": "replicas" if world > 1 else "single",
                   "positions": "%d consecutive decode steps ending at context %d" % (args.steps, T_last),
                   "l2": "inputs larger than L2 (a step reads ~3.4 GB of compressed keys and KV)",
                   "timing": "CUDA graph replay, CUDA events on the launching stream, max over ranks"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": dk["gbs"], "peak": hbm, "unit": "GB/s",
                     "frac": dk["frac"], "peak_source": peak_src + " hbm_gbs (burst copy)",
                     "traffic": ncu_traffic(dom), "alg_bytes_per_launch": dk["alg_bytes"],
                     "launch_us": dk["us"]},
        "kernels": kernels,
        # the whole step against HBM: every layer's selection and attention bytes over the step
        "select_attn_frac": {"bytes_per_step": n * (sel_b + att_b), "gbs": n * (sel_b + att_b) / (ms * 1e-3) / 1e9,
                             "peak": hbm, "frac": n * (sel_b + att_b) / (ms * 1e-3) / 1e9 / hbm},
        "e2e": {"value": replica_throughput(world, BATCH, e2e_steps, e2e_elapsed), "unit": "tok/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * launches_per_step,
        "device_error_flags": dev_err,
        "clocks": clk,
    }
    if offload is not None:
        line["offload"] = offload
    if ab is not None:
        line["selector_ab"] = ab
    if pf is not None:
        line["prefill"] = pf
    if cpu is not None:
        per_step, cores, desc = cpu
        line["cpu_baseline"] = {"value": BATCH / per_step, "unit": "tok/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
        if cpu_all is not None:
            pa, ca, da = cpu_all
            line["cpu_baseline"]["all_cores"] = {"value": BATCH / pa, "unit": "tok/s", "cores": ca, "sample": da}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
