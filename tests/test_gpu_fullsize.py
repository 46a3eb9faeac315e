"""Parity at the workloads' full sizes.

* One 8B-shaped layer with its KV resident, decoded at context 32768 for batch 1, 4 and 16:
  forecast projection 4096 -> 256, top-32 blocks plus the forced ones, 16 planted blocks per
  (sequence, group). Every selection and every attention output is compared with the oracle.
* The 32-layer, batch-16, context-131072 stack exactly as the benchmark builds and launches it
  (the same builder, the same launches, one step replayed from a CUDA graph):
  the oracle recomputes a sample of (layer, sequence, group) units one at a time from the
  same inputs, copied off the device before the step runs.
* The baseline multi-head selector at context 131072 for batch 1 and 16: sampled units'
  compressed keys (bit for bit) and selections.
* The offloaded step at batch 64, context 131072 (layer 0 resident, layers 1 and 2 in pinned
  host memory, the streams layout with its gather stream): sampled units' selections, the
  gathered blocks byte for byte, and attention outputs.
Every sampled unit's attention is checked over the GPU's own selection, which at a near-tie
may be another valid choice than the oracle's.
"""
import numpy as np
import pytest
import torch

import synth

from oracle import sparda_oracle as O
from tests.parity import check_attention, check_selection, to64
from tests.test_gpu_stack import make_stack_case, oracle_step, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sb(cuda_ok):
    from block_sparse_attention_forecast_gb300 import build
    build.build()
    import block_sparse_attention_forecast_gb300.binding as b
    b.sparda_device_error(clear=True)
    return b


@pytest.mark.parametrize("B", [1, 4, 16])
def test_one_layer_at_context_32768(sb, B):
    T = max_ctx = 32768
    shape, stack, inputs = make_stack_case(sb, 23 + B, 1, B, T, 32, max_ctx, 4096, 16)
    sel, out, S = oracle_step(inputs, 1, B, T, 32)
    stack.capture()
    stack.out.zero_()
    stack.idx.fill_(-7)
    stack.run()
    torch.cuda.synchronize()
    same = compare(stack, sel, out, S, 1, B, T, 32, inputs)
    assert same >= B * 2 * 3 // 4
    assert sb.sparda_device_error(clear=True) == 0


# (layer, sequence, group) units the oracle recomputes: first, second, middle and last layers
SAMPLED_UNITS = [(0, 0, 0), (0, 15, 1), (1, 3, 0), (1, 8, 1), (2, 5, 1), (13, 11, 0), (16, 0, 1),
                 (22, 9, 0), (30, 14, 1), (31, 2, 0), (31, 7, 1), (31, 15, 0)]


def test_benchmark_stack_sampled_units(sb):
    import bench
    device = "cuda:0"
    T = bench.CTX
    shape, stack, T0 = bench.build_workload(device, 0, 1)
    assert T0 == T and stack.mode == "pipelined"
    # the oracle's inputs, taken before the step writes token T-1
    units = {}
    for (L, b, g) in SAMPLED_UNITS:
        Wsel, hsel = (stack.W_self0, stack.h[0, b]) if L == 0 else (stack.W_next[L - 1], stack.h[L - 1, b])
        units[L, b, g] = dict(
            K=to64(stack.layers[L].k[b, g]), V=to64(stack.layers[L].v[b, g]), W=to64(Wsel), h=to64(hsel),
            q=to64(stack.q[L, b, 16 * g:16 * g + 16]), kn=to64(stack.k_new[L, b, g]),
            vn=to64(stack.v_new[L, b, g]))
    stack.capture()                  # one eager step, then the graph the benchmark replays
    stack.seq_len.fill_(T)
    stack.out.zero_()
    stack.idx.fill_(-7)
    stack.cnt.fill_(-7)
    stack.run()
    torch.cuda.synchronize()
    assert sb.sparda_device_error(clear=True) == 0
    idx, cnt = stack.idx.cpu().numpy(), stack.cnt.cpu().numpy()
    same = 0
    for (L, b, g), u in units.items():
        K, V = u["K"], u["V"]
        K[T - 1], V[T - 1] = u["kn"], u["vn"]
        f = O.forecast_project(u["W"], u["h"]).reshape(2, 128)[g]
        sel, S = O.forecast_select_one(K, f, T, bench.TOPK, return_scores=True)
        check_selection(idx[L, b, g], cnt[L, b, g], S, T, bench.TOPK)
        mine = [int(j) for j in idx[L, b, g, :cnt[L, b, g]]]
        same += mine == sel
        # the attention over the GPU's own selection: the oracle's where they agree, else the
        # other valid choice at a near-tie
        o_ref = O.block_sparse_attention(u["q"], K, V, mine, T)
        check_attention(to64(stack.out[L, b, 16 * g:16 * g + 16]), o_ref)
    assert same >= len(units) * 3 // 4
    del stack
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------------------
# the baseline multi-head selector at context 131072 (the selector A/B's context)
@pytest.mark.parametrize("B,units", [(1, [(0, 0), (0, 1)]), (16, [(0, 0), (3, 1), (7, 0), (12, 1), (15, 0), (15, 1)])])
def test_multihead_select_at_context_131072(sb, B, units):
    T = 131072
    shape = sb.Shape(n_groups=2, topk=32, max_ctx=T, max_batch=B)
    layer = sb.LayerKV.empty(shape)
    layer.k.copy_(synth.normal_bf16_device(layer.k.shape, 71 + B, "cuda"))
    layer.v.zero_()
    sb.sparda_compress_keys(shape, layer, torch.full((B,), T - 1, dtype=torch.int32, device="cuda"), B)
    q = synth.normal_bf16_device((B, 32, 128), 72 + B, "cuda")
    seq = torch.full((B,), T, dtype=torch.int32, device="cuda")
    idx = torch.full((B, 2, 34), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, 2), -7, dtype=torch.int32, device="cuda")
    ws = sb.workspace(shape, B, sb.WS_MULTIHEAD)
    sb.sparda_multihead_select(shape, layer.ck, q, seq, B, idx, cnt, ws)
    torch.cuda.synchronize()
    assert sb.sparda_device_error(clear=True) == 0
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    W = O.num_windows(T - 1)
    for b, g in units:
        ck = O.compress_keys(to64(layer.k[b, g, :T - 1]), W)
        assert np.array_equal(ck, to64(layer.ck[b, g, :W]))
        S = O.pool_to_blocks(O.multihead_scores(to64(q[b, 16 * g:16 * g + 16]), ck), (T - 1) // 64 + 1)
        check_selection(idx[b, g], cnt[b, g], S, T, 32)
    del layer, ws
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------------------
# the offloaded step at batch 64, context 131072: layer 0 resident, layers 1 and 2 with their
# K/V in pinned host memory, gathered over the host link on the gather stream
OFFLOAD_UNITS = [(0, 0, 0), (0, 63, 1), (1, 0, 1), (1, 17, 0), (1, 40, 1), (1, 63, 0), (2, 5, 0), (2, 33, 1),
                 (2, 62, 1)]


def test_offloaded_step_at_batch_64_context_131072(sb):
    from block_sparse_attention_forecast_gb300.step import DecodeStack
    n_layers, B, T, k, hidden, G, d = 3, 64, 131072, 32, 4096, 2, 128
    shape = sb.Shape(n_groups=G, topk=k, max_ctx=T, max_batch=B)
    dev = "cuda"
    W_self0 = synth.normal_bf16_device((G * d, hidden), 81, dev, std=0.02)
    W_next = [synth.normal_bf16_device((G * d, hidden), 82 + L, dev, std=0.02) for L in range(n_layers - 1)]
    h = synth.normal_bf16_device((n_layers, B, hidden), 85, dev)
    seq_c = torch.full((B,), T - 1, dtype=torch.int32, device=dev)
    layers = []
    for L in range(n_layers):
        Kd = synth.normal_bf16_device((B, G, T, d), 90 + L, dev)
        Vd = synth.normal_bf16_device((B, G, T, d), 95 + L, dev)
        if L == 0:
            layer = sb.LayerKV(Kd, Vd, torch.zeros((B, G, shape.w_cap, d), dtype=torch.bfloat16, device=dev))
        else:
            layer = sb.LayerKV.empty(shape, on_host=True)
            layer.k.copy_(Kd)
            layer.v.copy_(Vd)
            del Kd, Vd
        sb.sparda_compress_keys(shape, layer, seq_c, B)
        if L > 0:
            sb.fill_hot_from_host(layer, [T - 1] * B)
        layers.append(layer)
    stack = DecodeStack(shape, layers, W_self0, W_next, B)
    assert stack.mode == "streams"
    stack.h.copy_(h)
    stack.q.copy_(synth.normal_bf16_device(stack.q.shape, 86, dev))
    stack.k_new.copy_(synth.normal_bf16_device(stack.k_new.shape, 87, dev))
    stack.v_new.copy_(synth.normal_bf16_device(stack.v_new.shape, 88, dev))
    stack.seq_len.fill_(T)
    units = {}
    for (L, b, g) in OFFLOAD_UNITS:
        Wsel, hsel = (W_self0, h[0, b]) if L == 0 else (W_next[L - 1], h[L - 1, b])
        units[L, b, g] = dict(K=to64(layers[L].k[b, g]), V=to64(layers[L].v[b, g]), W=to64(Wsel), h=to64(hsel),
                              q=to64(stack.q[L, b, 16 * g:16 * g + 16]), kn=to64(stack.k_new[L, b, g]),
                              vn=to64(stack.v_new[L, b, g]))
    stack.enqueue()
    torch.cuda.synchronize()
    assert sb.sparda_device_error(clear=True) == 0
    idx, cnt = stack.idx.cpu().numpy(), stack.cnt.cpu().numpy()
    same = 0
    for (L, b, g), u in units.items():
        K, V = u["K"], u["V"]
        K[T - 1], V[T - 1] = u["kn"], u["vn"]
        f = O.forecast_project(u["W"], u["h"]).reshape(G, d)[g]
        sel, S = O.forecast_select_one(K, f, T, k, return_scores=True)
        check_selection(idx[L, b, g], cnt[L, b, g], S, T, k)
        mine = [int(j) for j in idx[L, b, g, :cnt[L, b, g]]]
        same += mine == sel
        if L > 0:
            # the gathered blocks, byte for byte, in the staging buffer of this layer
            tb = (T - 1) // 64
            sk, sv = stack.stage_k[L % 2][b, g].cpu(), stack.stage_v[L % 2][b, g].cpu()
            for s, j in enumerate(mine):
                if j not in (0, tb):
                    assert torch.equal(sk[s], layers[L].k[b, g, 64 * j:64 * j + 64]), (L, b, g, j)
                    assert torch.equal(sv[s], layers[L].v[b, g, 64 * j:64 * j + 64]), (L, b, g, j)
        o_ref = O.block_sparse_attention(u["q"], K, V, mine, T)
        check_attention(to64(stack.out[L, b, 16 * g:16 * g + 16]), o_ref)
    assert same >= len(units) * 3 // 4
    del stack, layers
    torch.cuda.empty_cache()
