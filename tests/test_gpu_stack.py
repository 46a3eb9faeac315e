"""A whole decode step of a small layer stack (forecast lookahead, layer 0 same-layer
forecast) through DecodeStack, eager and replayed from a CUDA graph, against the oracle's
decode_step on the same seeded inputs."""
import numpy as np
import pytest
import torch

import synth
from oracle import sparda_oracle as O
from tests.parity import check_attention, check_selection, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sb(cuda_ok):
    from block_sparse_attention_forecast_gb300 import build
    build.build()
    import block_sparse_attention_forecast_gb300.binding as b
    b.sparda_device_error(clear=True)
    return b


def make_stack_case(sb, seed, n_layers, B, T, topk, max_ctx, hidden, n_planted, offload=(), overlap=True,
                    mode="pipelined", block_cache=None):
    """Seeded caches holding tokens 0..T-2, the step's inputs, and forecast heads; planted
    blocks of each layer are shifted along the forecast (computed by the oracle) that selects
    that layer's blocks."""
    from block_sparse_attention_forecast_gb300.step import DecodeStack
    G, d = 2, 128
    shape = sb.Shape(n_groups=G, topk=topk, max_ctx=max_ctx, max_batch=B)
    W_self0 = synth.normal_bf16((G * d, hidden), seed, 100, std=0.02)
    W_next = [synth.normal_bf16((G * d, hidden), seed, 101, L, std=0.02) for L in range(n_layers - 1)]
    h = synth.normal_bf16((n_layers, B, hidden), seed, 102)
    q = synth.normal_bf16((n_layers, B, G * 16, d), seed, 103)
    kn = synth.normal_bf16((n_layers, B, G, d), seed, 104)
    vn = synth.normal_bf16((n_layers, B, G, d), seed, 105)
    nb = (T - 1) // 64 + 1
    Ks, Vs, layers = [], [], []
    for L in range(n_layers):
        K = synth.normal_bf16((B, G, max_ctx, d), seed, 200, L)
        V = synth.normal_bf16((B, G, max_ctx, d), seed, 201, L)
        Wsel, hsel = (W_self0, h[0]) if L == 0 else (W_next[L - 1], h[L - 1])
        for b in range(B):
            f = O.forecast_project(to64(Wsel), to64(hsel[b])).reshape(G, d)
            for g in range(G):
                synth.plant(K[b, g], synth.planted_blocks(seed, nb, n_planted, L, b, g), f[g])
        if L in offload:
            layer = sb.LayerKV.empty(shape, on_host=True)
            layer.k.copy_(K)
            layer.v.copy_(V)
            sb.fill_hot_from_host(layer, [T - 1] * B)
        else:
            layer = sb.LayerKV.empty(shape)
            layer.k.copy_(K.cuda())
            layer.v.copy_(V.cuda())
        sb.sparda_compress_keys(shape, layer, torch.full((B,), T - 1, dtype=torch.int32, device="cuda"), B)
        Ks.append(K)
        Vs.append(V)
        layers.append(layer)
    stack = DecodeStack(shape, layers, W_self0.cuda(), [w.cuda() for w in W_next], B, overlap=overlap,
                        mode=mode, block_cache=block_cache)
    stack.h.copy_(h.cuda())
    stack.q.copy_(q.cuda())
    stack.k_new.copy_(kn.cuda())
    stack.v_new.copy_(vn.cuda())
    stack.seq_len.fill_(T)
    inputs = dict(W_self0=W_self0, W_next=W_next, h=h, q=q, kn=kn, vn=vn, K=Ks, V=Vs)
    return shape, stack, inputs


def oracle_step(inputs, n_layers, B, T, topk):
    layers = [(to64(inputs["K"][L]), to64(inputs["V"][L])) for L in range(n_layers)]
    p = T - 1
    sel, out = O.decode_step(layers, to64(inputs["W_self0"]), [to64(w) for w in inputs["W_next"]],
                             [to64(inputs["h"][L]) for L in range(n_layers)],
                             [to64(inputs["q"][L]) for L in range(n_layers)],
                             [to64(inputs["kn"][L]) for L in range(n_layers)],
                             [to64(inputs["vn"][L]) for L in range(n_layers)], p, topk, 16)
    # block scores of every selection, for the near-tie rule
    S = {}
    for L in range(n_layers):
        Wsel, hsel = (inputs["W_self0"], inputs["h"][0]) if L == 0 else (inputs["W_next"][L - 1], inputs["h"][L - 1])
        for b in range(B):
            f = O.forecast_project(to64(Wsel), to64(hsel[b])).reshape(2, 128)
            for g in range(2):
                _, S[L, b, g] = O.forecast_select_one(layers[L][0][b, g], f[g], T, topk, return_scores=True)
    return sel, out, S


def compare(stack, sel, out, S, n_layers, B, T, topk, inputs):
    """Checks every unit's selection by the near-tie rule and every unit's attention: against
    the oracle's output where the selections agree, else against the oracle's attention over
    the GPU's own (valid) selection. Returns the number of units whose selections agree."""
    idx, cnt, o = stack.idx.cpu().numpy(), stack.cnt.cpu().numpy(), to64(stack.out)
    same = 0
    for L in range(n_layers):
        for b in range(B):
            for g in range(2):
                check_selection(idx[L, b, g], cnt[L, b, g], S[L, b, g], T, topk)
                mine = [int(j) for j in idx[L, b, g, :cnt[L, b, g]]]
                if mine == sel[L][b][g]:
                    same += 1
                    ref = out[L][b, 16 * g:16 * g + 16]
                else:
                    K, V = to64(inputs["K"][L][b, g]), to64(inputs["V"][L][b, g])
                    K[T - 1], V[T - 1] = to64(inputs["kn"][L][b, g]), to64(inputs["vn"][L][b, g])
                    ref = O.block_sparse_attention(to64(inputs["q"][L][b, 16 * g:16 * g + 16]), K, V, mine, T)
                check_attention(o[L, b, 16 * g:16 * g + 16], ref)
    return same


@pytest.mark.parametrize("mode", ["pipelined", "fused"])
@pytest.mark.parametrize("n_layers,B,T,topk,max_ctx,hidden", [
    (3, 2, 1500, 8, 2048, 256),
    (4, 3, 4097, 32, 8192, 4096),
])
def test_stack_step_eager_and_graph(sb, n_layers, B, T, topk, max_ctx, hidden, mode):
    shape, stack, inputs = make_stack_case(sb, 7, n_layers, B, T, topk, max_ctx, hidden, 8, mode=mode)
    sel, out, S = oracle_step(inputs, n_layers, B, T, topk)
    # eager
    stack.enqueue()
    torch.cuda.synchronize()
    same = compare(stack, sel, out, S, n_layers, B, T, topk, inputs)
    assert same >= n_layers * B * 2 * 3 // 4
    eager_out = stack.out.clone()
    eager_idx = stack.idx.clone()
    # the same step replayed from a CUDA graph: the step rewrites token T-1, so the result
    # is identical
    stack.out.zero_()
    stack.capture()
    stack.out.zero_()
    stack.run()
    torch.cuda.synchronize()
    assert torch.equal(stack.idx, eager_idx)
    assert torch.equal(stack.out, eager_out)
    assert sb.sparda_device_error(clear=True) == 0


@pytest.mark.parametrize("overlap", [True, False])
def test_offloaded_stack_step(sb, overlap):
    # layer 0 resident, layers 1..3 offloaded to pinned host memory; the gather of layer L+1
    # runs on its own stream, overlapped with layer L (or waited on at once)
    n_layers, B, T, topk, max_ctx, hidden = 4, 2, 2500, 8, 4096, 256
    shape, stack, inputs = make_stack_case(sb, 9, n_layers, B, T, topk, max_ctx, hidden, 8,
                                           offload={1, 2, 3}, overlap=overlap)
    sel, out, S = oracle_step(inputs, n_layers, B, T, topk)
    stack.enqueue()
    torch.cuda.synchronize()
    same = compare(stack, sel, out, S, n_layers, B, T, topk, inputs)
    assert same >= n_layers * B * 2 * 3 // 4
    eager_out, eager_idx = stack.out.clone(), stack.idx.clone()
    stack.capture()
    stack.out.zero_()
    stack.run()
    torch.cuda.synchronize()
    assert torch.equal(stack.idx, eager_idx)
    assert torch.equal(stack.out, eager_out)
    assert sb.sparda_device_error(clear=True) == 0


@pytest.mark.parametrize("B", [3, 17, 18])
def test_all_launch_modes_agree(sb, B):
    # the same step launched as two kernels per layer (prologue with the top-k +
    # attend-and-score), three (projection, append, attend-and-select) or one kernel per job
    # on two streams: the same arithmetic, bit-identical results. B = 17 is the largest batch
    # whose selection (34 sequence-groups) attend-and-score hands out from a queue; from
    # B = 18 (36) each selection CTA takes a fixed range instead.
    n_layers, T, topk, max_ctx, hidden = 4, 3001, 8, 4096, 256
    outs = []
    for mode in ("pipelined", "fused", "streams"):
        shape, stack, inputs = make_stack_case(sb, 11, n_layers, B, T, topk, max_ctx, hidden, 8, mode=mode)
        assert stack.mode == mode
        stack.enqueue()
        torch.cuda.synchronize()
        outs.append((stack.idx.clone(), stack.cnt.clone(), stack.out.clone()))
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            assert torch.equal(a, b)
    assert sb.sparda_device_error(clear=True) == 0


@pytest.mark.parametrize("call", ["score", "select"])
@pytest.mark.parametrize("B", [3, 18])
def test_back_to_back_attend_calls(sb, call, B):
    # Each attend-and-score / attend-and-select launch lets the next launch begin while it
    # runs, so calls directly after one another on a stream overlap (at these small shapes
    # the grids leave SMs free, so more than two may run at once). With a selection workspace
    # of its own for each call (the rule the header states), the calls give exactly what the
    # same calls give one at a time; in the attend-and-select chain each call's attention
    # reads the blocks the call before selected. B = 3 hands the selection out from a queue,
    # B = 18 in fixed ranges.
    n_layers, T, topk, max_ctx, hidden = 5, 4097, 32, 8192, 256
    shape, stack, _ = make_stack_case(sb, 37, n_layers, B, T, topk, max_ctx, hidden, 8)
    stack.enqueue()                                  # idx, cnt and forecasts of every layer
    torch.cuda.synchronize()
    idx0, cnt0 = stack.idx.clone(), stack.cnt.clone()
    off = sb.sparda_block_scores_offset(shape)
    n_sc = B * shape.n_groups * (max_ctx // 64) * 4

    def run(sync):
        stack.idx.copy_(idx0)
        stack.cnt.copy_(cnt0)
        stack.out.zero_()
        torch.cuda.synchronize()
        ws = [sb.workspace(shape, B, sb.WS_SELECT) for _ in range(n_layers - 1)]
        ws_attn = sb.workspace(shape, B, sb.WS_ATTN)
        for L in range(n_layers - 1):
            w = ws[L]
            if call == "score":
                sb.sparda_attend_and_score(shape, stack.layers[L], stack.q[L], stack.idx[L], stack.cnt[L], stack.out[L],
                                           ws_attn, stack.layers[L + 1].ck, stack.f[L + 1], w, stack.seq_len, B)
            else:
                sb.sparda_attend_and_select(shape, stack.layers[L], stack.q[L], stack.idx[L], stack.cnt[L],
                                            stack.out[L], ws_attn, stack.layers[L + 1].ck, stack.f[L + 1],
                                            stack.idx[L + 1], stack.cnt[L + 1], w, stack.seq_len, B)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        scores = torch.stack([w[off:off + n_sc] for w in ws])
        return stack.idx.clone(), stack.cnt.clone(), stack.out[:n_layers - 1].clone(), scores

    ref, got = run(True), run(False)
    for a, b in zip(ref, got):
        assert torch.equal(a, b)
    assert sb.sparda_device_error(clear=True) == 0


@pytest.mark.parametrize("mode", ["pipelined", "fused"])
def test_single_layer_stack(sb, mode):
    # one layer: layer 0's own selection, its prologue without a top-k or projection, its
    # attention alone
    shape, stack, inputs = make_stack_case(sb, 13, 1, 2, 2000, 8, 2048, 256, 8, mode=mode)
    sel, out, S = oracle_step(inputs, 1, 2, 2000, 8)
    stack.enqueue()
    torch.cuda.synchronize()
    assert compare(stack, sel, out, S, 1, 2, 2000, 8, inputs) >= 3
    assert sb.sparda_device_error(clear=True) == 0


@pytest.mark.parametrize("mode,offload", [("pipelined", ()), ("fused", ()), ("streams", ()), ("streams", (2, 3))])
def test_host_io_step(sb, mode, offload):
    # inputs from pinned host memory and outputs back to it, copied inside the step on the
    # I/O stream: the same results as with the inputs already on the device, eager and from a
    # CUDA graph
    n_layers, B, T, topk, max_ctx, hidden = 6, 2, 2500, 8, 4096, 256
    shape, stack, inputs = make_stack_case(sb, 15, n_layers, B, T, topk, max_ctx, hidden, 8, mode=mode,
                                           offload=set(offload))
    stack.enqueue()
    torch.cuda.synchronize()
    ref_out, ref_idx = stack.out.clone(), stack.idx.clone()
    names = ("h", "q", "k_new", "v_new")
    host_in = stack.pinned_inputs()
    for n in names:
        host_in[n].copy_(getattr(stack, n).cpu())
    host_out = torch.zeros_like(stack.out, device="cpu").pin_memory()
    with pytest.raises(ValueError):
        stack.attach_host_io({**host_in, "q": host_in["q"].clone()}, host_out)   # not a view of packed
    with pytest.raises(ValueError):
        stack.attach_host_io({n: host_in[n] for n in names}, host_out)          # no packed buffer
    with pytest.raises(ValueError):
        stack.attach_host_io(host_in, host_out.clone())                        # output not pinned
    stack.attach_host_io(host_in, host_out)
    assert stack.io_bytes() == (host_in["packed"].numel(), stack.out.numel() * 2)
    assert host_in["packed"].numel() >= sum(getattr(stack, n).numel() * 2 for n in names)

    def clear():
        for n in names:
            getattr(stack, n).zero_()
        stack.out.zero_()
        stack.idx.fill_(-1)
        host_out.zero_()
        torch.cuda.synchronize()

    clear()
    stack.enqueue()
    torch.cuda.synchronize()
    assert torch.equal(host_out, ref_out.cpu())
    assert torch.equal(stack.idx, ref_idx)
    clear()
    stack.capture()
    clear()
    stack.run()
    torch.cuda.synchronize()
    assert torch.equal(host_out, ref_out.cpu())
    assert torch.equal(stack.idx, ref_idx)
    stack.attach_host_io(None, None)
    assert stack.io_bytes() == (0, 0)
    assert sb.sparda_device_error(clear=True) == 0
