"""Chunked prefill through the C ABI against the oracle: the Forecast and the baseline
multi-head chunk selections (block indices, by the near-tie rule) and the causal block-sparse
prefill attention (element-wise, over the GPU's own selections), on ragged prompts that span
several chunk tiles and at context 32768 on sampled chunks and tokens."""
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


def _prompt(sb, seed, T_list, k, max_ctx):
    B, G, H, d = len(T_list), 2, 16, 128
    shape = sb.Shape(n_groups=G, topk=k, max_ctx=max_ctx, max_batch=B)
    layer = sb.LayerKV.empty(shape)
    layer.k.copy_(synth.normal_bf16((B, G, max_ctx, d), seed, 1).cuda())
    layer.v.copy_(synth.normal_bf16((B, G, max_ctx, d), seed, 2).cuda())
    q = synth.normal_bf16((B, max_ctx, G * H, d), seed, 3).cuda()
    f = synth.normal_bf16((B, max_ctx, G, d), seed, 4).cuda()
    seq = torch.tensor(T_list, dtype=torch.int32, device="cuda")
    sb.sparda_compress_keys(shape, layer, seq, B)
    return shape, layer, q, f, seq


def _select(sb, shape, which, layer, qf, seq, B):
    nc = shape.max_ctx // 64
    idx = torch.full((B, 2, nc, shape.kslots), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, 2, nc), -7, dtype=torch.int32, device="cuda")
    ws = sb.workspace(shape, B, sb.WS_PREFILL)
    fn = sb.sparda_prefill_forecast_select if which == "forecast" else sb.sparda_prefill_multihead_select
    fn(shape, layer.ck, qf, seq, B, idx, cnt, ws)
    torch.cuda.synchronize()
    assert sb.sparda_device_error(clear=True) == 0
    return idx, cnt


def _check_chunks(idx, cnt, b, g, T, k, ck, chunks, queries, which):
    for c in chunks:
        if which == "forecast":
            s = O.prefill_forecast_scores(queries(c), ck, c)
        else:
            s = O.prefill_multihead_scores(queries(c), ck, c)
        S = O.pool_to_blocks(s, c + 1)
        check_selection(idx[b, g, c], cnt[b, g, c], S, 64 * c + 1, k)


@pytest.mark.parametrize("which", ["forecast", "multihead"])
@pytest.mark.parametrize("T_list,k,max_ctx", [([1500, 700, 64, 1], 4, 2048), ([2049, 1111], 8, 4096)])
def test_prefill_selection(sb, which, T_list, k, max_ctx):
    shape, layer, q, f, seq = _prompt(sb, 31 + k, T_list, k, max_ctx)
    B = len(T_list)
    idx, cnt = _select(sb, shape, which, layer, f if which == "forecast" else q, seq, B)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    for b, T in enumerate(T_list):
        nc = O.prefill_num_chunks(T)
        assert (cnt[b, :, nc:] == 0).all() and (idx[b, :, nc:] == -1).all()
        for g in range(2):
            ck = O.compress_keys(to64(layer.k[b, g, :T]), O.num_windows(T))
            assert np.array_equal(ck, to64(layer.ck[b, g, :O.num_windows(T)]))
            if which == "forecast":
                queries = lambda c: to64(f[b, 64 * c:min(64 * c + 64, T), g])
            else:
                queries = lambda c: to64(q[b, 64 * c:min(64 * c + 64, T), 16 * g:16 * g + 16])
            _check_chunks(idx, cnt, b, g, T, k, ck, range(nc), queries, which)


@pytest.mark.parametrize("T_list,k,max_ctx", [([1500, 700, 64, 1], 4, 2048), ([2049, 130], 8, 4096)])
def test_prefill_attention(sb, T_list, k, max_ctx):
    shape, layer, q, f, seq = _prompt(sb, 41 + k, T_list, k, max_ctx)
    B = len(T_list)
    idx, cnt = _select(sb, shape, "forecast", layer, f, seq, B)
    out = torch.full((B, max_ctx, 32, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    sb.sparda_prefill_attn(shape, layer, q, idx, cnt, seq, B, out)
    torch.cuda.synchronize()
    assert sb.sparda_device_error(clear=True) == 0
    idx, cnt, o = idx.cpu().numpy(), cnt.cpu().numpy(), out.float().cpu().numpy()
    for b, T in enumerate(T_list):
        assert (o[b, T:] == 7.0).all()                       # nothing written past the prompt
        for g in range(2):
            sel = [[int(j) for j in idx[b, g, c, :cnt[b, g, c]]] for c in range(O.prefill_num_chunks(T))]
            ref = O.prefill_block_sparse_attention(to64(q[b, :T, 16 * g:16 * g + 16]), to64(layer.k[b, g]),
                                                   to64(layer.v[b, g]), sel, T)
            for t in range(T):
                check_attention(o[b, t, 16 * g:16 * g + 16], ref[t])


def test_prefill_attention_with_every_block_is_dense_causal(sb):
    # k at least the number of candidate blocks: every chunk keeps all blocks up to its own,
    # and the block-sparse prefill is dense causal attention
    T, max_ctx = 900, 1024
    shape, layer, q, f, seq = _prompt(sb, 51, [T], 62, max_ctx)
    idx, cnt = _select(sb, shape, "forecast", layer, f, seq, 1)
    assert [int(x) for x in cnt[0, 0, :15].cpu()] == [c + 1 for c in range(15)]
    out = torch.zeros((1, max_ctx, 32, 128), dtype=torch.bfloat16, device="cuda")
    sb.sparda_prefill_attn(shape, layer, q, idx, cnt, seq, 1, out)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    for g in range(2):
        ref = O.dense_causal_prefill_attention(to64(q[0, :T, 16 * g:16 * g + 16]), to64(layer.k[0, g]),
                                               to64(layer.v[0, g]), T)
        for t in range(T):
            check_attention(o[0, t, 16 * g:16 * g + 16], ref[t])


SAMPLED_CHUNKS = [0, 1, 2, 37, 255, 400, 511]


def test_prefill_at_context_32768_sampled(sb):
    T = max_ctx = 32768
    k = 32
    shape = sb.Shape(n_groups=2, topk=k, max_ctx=max_ctx, max_batch=1)
    layer = sb.LayerKV.empty(shape)
    layer.k.copy_(synth.normal_bf16_device(layer.k.shape, 61, "cuda"))
    layer.v.copy_(synth.normal_bf16_device(layer.v.shape, 62, "cuda"))
    q = synth.normal_bf16_device((1, max_ctx, 32, 128), 63, "cuda")
    f = synth.normal_bf16_device((1, max_ctx, 2, 128), 64, "cuda")
    seq = torch.full((1,), T, dtype=torch.int32, device="cuda")
    sb.sparda_compress_keys(shape, layer, seq, 1)
    res = {w: [x.cpu().numpy() for x in _select(sb, shape, w, layer, f if w == "forecast" else q, seq, 1)]
           for w in ("forecast", "multihead")}
    idx_t = torch.from_numpy(res["forecast"][0]).cuda()
    cnt_t = torch.from_numpy(res["forecast"][1]).cuda()
    out = torch.zeros((1, max_ctx, 32, 128), dtype=torch.bfloat16, device="cuda")
    sb.sparda_prefill_attn(shape, layer, q, idx_t, cnt_t, seq, 1, out)
    torch.cuda.synchronize()
    assert sb.sparda_device_error(clear=True) == 0
    for g in range(2):
        K, V = to64(layer.k[0, g]), to64(layer.v[0, g])
        ck = to64(layer.ck[0, g])
        for which, (idx, cnt) in res.items():
            if which == "forecast":
                queries = lambda c: to64(f[0, 64 * c:64 * c + 64, g])
            else:
                queries = lambda c: to64(q[0, 64 * c:64 * c + 64, 16 * g:16 * g + 16])
            _check_chunks(idx, cnt, 0, g, T, k, ck, SAMPLED_CHUNKS, queries, which)
        idx, cnt = res["forecast"]
        for c in SAMPLED_CHUNKS:
            sel = [int(j) for j in idx[0, g, c, :cnt[0, g, c]]]
            for t in (64 * c, 64 * c + 31, 64 * c + 63):
                toks = O.selected_tokens(sel, t + 1)
                ref = O.block_sparse_attention(to64(q[0, t, 16 * g:16 * g + 16]), K, V, sel, t + 1)
                assert toks[-1] == t
                check_attention(out[0, t, 16 * g:16 * g + 16].float().cpu().numpy(), ref)


def test_prefill_attention_when_later_blocks_dominate(sb):
    """Keys of the later blocks scaled up four-fold: every chunk's later blocks carry far larger
    logits than block 0, so the running maximum of the online softmax must move (and the
    partial output be rescaled) part-way through the blocks."""
    T_list, k, max_ctx = [1100, 777], 6, 2048
    shape, layer, q, f, seq = _prompt(sb, 57, T_list, k, max_ctx)
    layer.k[:, :, 256:] *= 4
    B = len(T_list)
    idx, cnt = _select(sb, shape, "forecast", layer, f, seq, B)
    out = torch.zeros((B, max_ctx, 32, 128), dtype=torch.bfloat16, device="cuda")
    sb.sparda_prefill_attn(shape, layer, q, idx, cnt, seq, B, out)
    torch.cuda.synchronize()
    assert sb.sparda_device_error(clear=True) == 0
    idx, cnt, o = idx.cpu().numpy(), cnt.cpu().numpy(), out.float().cpu().numpy()
    for b, T in enumerate(T_list):
        for g in range(2):
            sel = [[int(j) for j in idx[b, g, c, :cnt[b, g, c]]] for c in range(O.prefill_num_chunks(T))]
            ref = O.prefill_block_sparse_attention(to64(q[b, :T, 16 * g:16 * g + 16]), to64(layer.k[b, g]),
                                                   to64(layer.v[b, g]), sel, T)
            for t in range(T):
                check_attention(o[b, t, 16 * g:16 * g + 16], ref[t])


def test_prefill_selection_at_the_largest_context_shape(sb):
    """max_ctx 262144: the baseline selector's window sums take the room of a ring stage (two
    stages instead of three); a 5000-token prompt, every chunk checked, both selectors."""
    max_ctx, T, k = 262144, 5000, 8
    shape = sb.Shape(n_groups=2, topk=k, max_ctx=max_ctx, max_batch=1)
    layer = sb.LayerKV.empty(shape)
    layer.k.copy_(synth.normal_bf16_device(layer.k.shape, 81, "cuda"))
    layer.v.copy_(synth.normal_bf16_device(layer.v.shape, 82, "cuda"))
    q = synth.normal_bf16_device((1, max_ctx, 32, 128), 83, "cuda")
    f = synth.normal_bf16_device((1, max_ctx, 2, 128), 84, "cuda")
    seq = torch.full((1,), T, dtype=torch.int32, device="cuda")
    sb.sparda_compress_keys(shape, layer, seq, 1)
    nc = O.prefill_num_chunks(T)
    for which in ("forecast", "multihead"):
        idx, cnt = _select(sb, shape, which, layer, f if which == "forecast" else q, seq, 1)
        idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
        assert (cnt[0, :, nc:] == 0).all()
        for g in range(2):
            ck = O.compress_keys(to64(layer.k[0, g, :T]), O.num_windows(T))
            if which == "forecast":
                queries = lambda c: to64(f[0, 64 * c:min(64 * c + 64, T), g])
            else:
                queries = lambda c: to64(q[0, 64 * c:min(64 * c + 64, T), 16 * g:16 * g + 16])
            _check_chunks(idx, cnt, 0, g, T, k, ck, range(nc), queries, which)
