"""Parity of each libsparda kernel with the fp64 oracle, on small seeded inputs that span
several tiles and ragged tails. Every call goes through the C ABI (the ctypes binding)."""
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


def _no_device_error(sb):
    assert sb.sparda_device_error(clear=True) == 0


# ------------------------------------------------------------------ compressed keys
@pytest.mark.parametrize("T_list", [[1000, 33, 64], [31, 32, 47, 48], [1024, 1023, 999, 512]])
def test_compress_keys_bit_exact(sb, T_list):
    B = len(T_list)
    shape = sb.Shape(max_ctx=1024, max_batch=B, topk=8)
    layer = sb.LayerKV.empty(shape)
    K = synth.normal_bf16((B, 2, 1024, 128), 11, B)
    layer.k.copy_(K.cuda())
    layer.v.zero_()
    seq = torch.tensor(T_list, dtype=torch.int32, device="cuda")
    sb.sparda_compress_keys(shape, layer, seq, B)
    torch.cuda.synchronize()
    ck = to64(layer.ck)
    for b, T in enumerate(T_list):
        for g in range(2):
            W = O.num_windows(T)
            want = O.compress_keys(to64(K[b, g]), W)
            assert np.array_equal(ck[b, g, :W], want), (b, g, T)
    _no_device_error(sb)


def test_append_tokens_and_windows(sb):
    B, steps, T0 = 3, 70, [100, 37, 500]
    shape = sb.Shape(max_ctx=1024, max_batch=B, topk=8)
    layer = sb.LayerKV.empty(shape)
    K = synth.normal_bf16((B, 2, 1024, 128), 12, 1)
    V = synth.normal_bf16((B, 2, 1024, 128), 12, 2)
    layer.k.copy_(K.cuda())
    layer.v.copy_(V.cuda())
    seq = torch.tensor(T0, dtype=torch.int32, device="cuda")
    sb.sparda_compress_keys(shape, layer, seq, B)
    Kref, Vref = to64(K), to64(V)
    for s in range(steps):
        T = [t + s + 1 for t in T0]                      # the new token sits at T - 1
        kn = synth.normal_bf16((B, 2, 128), 13, s, 1)
        vn = synth.normal_bf16((B, 2, 128), 13, s, 2)
        seq.copy_(torch.tensor(T, dtype=torch.int32))
        sb.sparda_append_kv(shape, layer, kn.cuda(), vn.cuda(), seq, B)
        for b in range(B):
            Kref[b, :, T[b] - 1] = to64(kn[b])
            Vref[b, :, T[b] - 1] = to64(vn[b])
    torch.cuda.synchronize()
    k_gpu, v_gpu, ck = to64(layer.k), to64(layer.v), to64(layer.ck)
    for b in range(B):
        T = T0[b] + steps
        assert np.array_equal(k_gpu[b, :, :T], Kref[b, :, :T])
        assert np.array_equal(v_gpu[b, :, :T], Vref[b, :, :T])
        for g in range(2):
            W = O.num_windows(T)
            assert np.array_equal(ck[b, g, :W], O.compress_keys(Kref[b, g], W)), (b, g)
    _no_device_error(sb)


# ------------------------------------------------------------------ forecast projection
@pytest.mark.parametrize("B,rows,hidden", [(1, 256, 4096), (5, 256, 4096), (16, 256, 4096),
                                           (20, 64, 96), (64, 256, 4096)])
def test_forecast_project(sb, B, rows, hidden):
    W = synth.normal_bf16((rows, hidden), 21, B, std=0.02)
    h = synth.normal_bf16((B, hidden), 22, B)
    f = torch.empty((B, rows), dtype=torch.bfloat16, device="cuda")
    sb.sparda_forecast_project(W.cuda(), h.cuda(), f)
    torch.cuda.synchronize()
    got = to64(f)
    Wd, hd = to64(W), to64(h)
    exact = hd @ Wd.T                                    # unrounded float64 products
    want = O.bf16_round(exact)
    diff = got != want
    # A float32 sum may round to the other bf16 neighbour only when the exact value sits
    # within float32 accumulation error of the midpoint between the two (and then the two
    # values are neighbours, since the exact value lies between them).
    if diff.any():
        lo, hi = np.minimum(got, want)[diff], np.maximum(got, want)[diff]
        mid = (lo + hi) / 2
        e = exact[diff]
        assert np.all(np.abs(e - mid) <= 2e-4 * np.abs(e) + 1e-6), "non-midpoint rounding difference"
    assert diff.mean() < 0.01


# ------------------------------------------------------------------ forecast selector
def _select_case(sb, K, f, T_list, k, max_ctx):
    B = len(T_list)
    shape = sb.Shape(max_ctx=max_ctx, max_batch=B, topk=k)
    ck = torch.zeros((B, 2, shape.w_cap, 128), dtype=torch.bfloat16)
    Sref = {}
    for b, T in enumerate(T_list):
        for g in range(2):
            W = O.num_windows(T - 1)
            c = O.compress_keys(to64(K[b, g]), W)
            ck[b, g, :W] = torch.from_numpy(c).to(torch.bfloat16)
            s = O.forecast_scores(c, to64(f[b, g]))
            Sref[b, g] = O.pool_to_blocks(s, (T - 1) // 64 + 1)
    seq = torch.tensor(T_list, dtype=torch.int32, device="cuda")
    idx = torch.full((B, 2, k + 2), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, 2), -7, dtype=torch.int32, device="cuda")
    ws = sb.workspace(shape, B, sb.WS_SELECT)
    for rep in range(2):                                 # the workspace is reusable as left
        sb.sparda_forecast_select(shape, ck.cuda(), f.cuda(), seq, B, idx, cnt, ws)
        torch.cuda.synchronize()
        unique = 0
        for b, T in enumerate(T_list):
            for g in range(2):
                unique += check_selection(idx[b, g].cpu().numpy(), cnt[b, g].item(), Sref[b, g], T, k)
    _no_device_error(sb)
    return unique


def test_select_tiny_planted(sb):
    # batch 1, context 4096, k = 8, 8 planted blocks per group shifted along the forecast
    for seed in range(3):
        case = synth.tiny_case(seed)
        unique = _select_case(sb, case["K"], case["f"], [4096], 8, 4096)
        assert unique >= 1


@pytest.mark.parametrize("T_list,k,max_ctx", [
    ([1, 2, 64, 65], 8, 1024),                # no candidates: forced blocks only
    ([129, 200, 256, 257], 8, 1024),          # fewer candidates than k
    ([4096, 4000, 1000, 3333], 8, 4096),
    ([8192, 7777, 5000, 6401], 32, 8192),     # k = 32, ragged tails
    ([16384, 9999], 62, 16384),               # the largest k
    ([140000, 131073], 32, 262144),           # the largest context: 16 scores per top-k thread
])
def test_select_ragged(sb, T_list, k, max_ctx):
    B = len(T_list)
    K = synth.normal_bf16((B, 2, max_ctx, 128), 31, B, k)
    f = synth.normal_bf16((B, 2, 128), 32, B, k)
    _select_case(sb, K, f, T_list, k, max_ctx)


def test_select_ties_break_to_lower_block(sb):
    # Every window identical -> every candidate block scores the same; the selection must be
    # the k lowest candidate indices.
    T, k = 2048, 8
    K = torch.ones((1, 2, T, 128), dtype=torch.bfloat16) * 0.5
    f = torch.ones((1, 2, 128), dtype=torch.bfloat16)
    shape = sb.Shape(max_ctx=T, max_batch=1, topk=k)
    layer = sb.LayerKV.empty(shape)
    layer.k.copy_(K.cuda())
    seq = torch.tensor([T], dtype=torch.int32, device="cuda")
    sb.sparda_compress_keys(shape, layer, torch.tensor([T - 1], dtype=torch.int32, device="cuda"), 1)
    idx = torch.zeros((1, 2, k + 2), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    ws = sb.workspace(shape, 1, sb.WS_SELECT)
    sb.sparda_forecast_select(shape, layer.ck, f.cuda(), seq, 1, idx, cnt, ws)
    torch.cuda.synchronize()
    for g in range(2):
        assert idx[0, g].tolist() == [0, 1, 2, 3, 4, 5, 6, 7, 8, 31]
    _no_device_error(sb)


# ------------------------------------------------------------------ attention
@pytest.mark.parametrize("T_list,k,max_ctx", [
    ([4096], 8, 4096),
    ([1, 63, 64, 65], 8, 1024),
    ([3000, 1500, 4095], 8, 4096),
    ([8192, 7000], 32, 8192),
    ([16384], 62, 16384),
])
def test_sparse_attention(sb, T_list, k, max_ctx):
    B = len(T_list)
    shape = sb.Shape(max_ctx=max_ctx, max_batch=B, topk=k)
    K = synth.normal_bf16((B, 2, max_ctx, 128), 41, B, k)
    V = synth.normal_bf16((B, 2, max_ctx, 128), 42, B, k)
    q = synth.normal_bf16((B, 32, 128), 43, B, k)
    f = synth.normal_bf16((B, 2, 128), 44, B, k)
    layer = sb.LayerKV.empty(shape)
    layer.k.copy_(K.cuda())
    layer.v.copy_(V.cuda())
    idx = torch.full((B, 2, k + 2), -1, dtype=torch.int32)
    cnt = torch.zeros((B, 2), dtype=torch.int32)
    sels = {}
    for b, T in enumerate(T_list):
        for g in range(2):
            sel = O.forecast_select_one(to64(K[b, g]), to64(f[b, g]), T, k)
            sels[b, g] = sel
            idx[b, g, :len(sel)] = torch.tensor(sel, dtype=torch.int32)
            cnt[b, g] = len(sel)
    out = torch.full((B, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = sb.workspace(shape, B, sb.WS_ATTN)
    seq = torch.tensor(T_list, dtype=torch.int32, device="cuda")
    for rep in range(2):
        sb.sparda_sparse_decode_attn(shape, layer, q.cuda(), idx.cuda(), cnt.cuda(), seq, B, out, ws)
        torch.cuda.synchronize()
        o = to64(out)
        for b, T in enumerate(T_list):
            for g in range(2):
                ref = O.block_sparse_attention(to64(q[b, 16 * g:16 * g + 16]), to64(K[b, g]),
                                               to64(V[b, g]), sels[b, g], T)
                check_attention(o[b, 16 * g:16 * g + 16], ref)
    _no_device_error(sb)


# Batches whose groups split evenly over 2 to 8 CTAs run the merge of a group's partial
# results in one thread-block cluster (distributed shared memory); batch 5 splits its groups
# over 15 CTAs and merges through the workspace in two rounds. Ragged lengths give groups with
# fewer selected blocks than CTAs (empty partials), and k = 1 three slots per group.
@pytest.mark.parametrize("B,k,max_ctx", [(8, 32, 2048), (12, 16, 2048), (16, 32, 4096), (24, 8, 1024),
                                         (32, 1, 1024), (5, 32, 4096)])
def test_sparse_attention_split_groups(sb, B, k, max_ctx):
    rng = np.random.default_rng(1000 + B)
    T_list = [int(x) for x in rng.integers(1, max_ctx + 1, size=B)]
    T_list[0], T_list[-1] = max_ctx, 1
    shape = sb.Shape(max_ctx=max_ctx, max_batch=B, topk=k)
    K = synth.normal_bf16((B, 2, max_ctx, 128), 71, B, k)
    V = synth.normal_bf16((B, 2, max_ctx, 128), 72, B, k)
    q = synth.normal_bf16((B, 32, 128), 73, B, k)
    layer = sb.LayerKV.empty(shape)
    layer.k.copy_(K.cuda())
    layer.v.copy_(V.cuda())
    idx = torch.full((B, 2, k + 2), -1, dtype=torch.int32)
    cnt = torch.zeros((B, 2), dtype=torch.int32)
    sels = {}
    for b, T in enumerate(T_list):
        nb = (T - 1) // 64 + 1
        for g in range(2):
            n = min(k + 2, nb) - int(rng.integers(0, 2))      # sometimes one slot short
            sel = sorted(int(x) for x in rng.choice(nb, size=max(n, 1), replace=False))
            sels[b, g] = sel
            idx[b, g, :len(sel)] = torch.tensor(sel, dtype=torch.int32)
            cnt[b, g] = len(sel)
    out = torch.full((B, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = sb.workspace(shape, B, sb.WS_ATTN)
    seq = torch.tensor(T_list, dtype=torch.int32, device="cuda")
    for rep in range(2):                      # the second call finds the workspace counters reset
        sb.sparda_sparse_decode_attn(shape, layer, q.cuda(), idx.cuda(), cnt.cuda(), seq, B, out, ws)
        torch.cuda.synchronize()
        o = to64(out)
        for b, T in enumerate(T_list):
            for g in range(2):
                ref = O.block_sparse_attention(to64(q[b, 16 * g:16 * g + 16]), to64(K[b, g]),
                                               to64(V[b, g]), sels[b, g], T)
                check_attention(o[b, 16 * g:16 * g + 16], ref)
    _no_device_error(sb)


# Calls issued back to back without a host synchronisation. Each attention launch lets the next
# launch begin at its start, so this checks the ordering the library keeps without a host wait:
# a second attention sharing the first one's workspace, a forecast selection (which may also
# begin early) rewriting the block indices the first attention read, and a third attention
# reading the new indices and writing the first one's output buffer. Batch 16 merges each
# group in a thread-block cluster, batch 5 through the workspace.
@pytest.mark.parametrize("B", [16, 5])
def test_attention_calls_back_to_back(sb, B):
    k, max_ctx = 16, 4096
    rng = np.random.default_rng(3000 + B)
    T_list = [int(x) for x in rng.integers(200, max_ctx + 1, size=B)]
    T_list[0] = max_ctx
    shape = sb.Shape(max_ctx=max_ctx, max_batch=B, topk=k)
    K = synth.normal_bf16((B, 2, max_ctx, 128), 81, B)
    V = synth.normal_bf16((B, 2, max_ctx, 128), 82, B)
    qs = [synth.normal_bf16((B, 32, 128), 83 + i, B) for i in range(3)]
    f = synth.normal_bf16((B, 2, 128), 86, B)
    layer = sb.LayerKV.empty(shape)
    layer.k.copy_(K.cuda())
    layer.v.copy_(V.cuda())
    seq = torch.tensor(T_list, dtype=torch.int32, device="cuda")
    sb.sparda_compress_keys(shape, layer, seq - 1, B)
    # two fixed selections (random block sets) for the first two calls
    sels = []
    idx_d, cnt_d = [], []
    for i in range(2):
        idx = torch.full((B, 2, k + 2), -1, dtype=torch.int32)
        cnt = torch.zeros((B, 2), dtype=torch.int32)
        sel_i = {}
        for b, T in enumerate(T_list):
            nb = (T - 1) // 64 + 1
            for g in range(2):
                sel = sorted(int(x) for x in rng.choice(nb, size=min(k + 2, nb), replace=False))
                sel_i[b, g] = sel
                idx[b, g, :len(sel)] = torch.tensor(sel, dtype=torch.int32)
                cnt[b, g] = len(sel)
        sels.append(sel_i)
        idx_d.append(idx.cuda())
        cnt_d.append(cnt.cuda())
    wa = sb.workspace(shape, B, sb.WS_ATTN)
    ws = sb.workspace(shape, B, sb.WS_SELECT)
    out1 = torch.full((B, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    out2 = torch.full((B, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    q_d = [q.cuda() for q in qs]
    torch.cuda.synchronize()
    sb.sparda_sparse_decode_attn(shape, layer, q_d[0], idx_d[0], cnt_d[0], seq, B, out1, wa)
    sb.sparda_sparse_decode_attn(shape, layer, q_d[1], idx_d[1], cnt_d[1], seq, B, out2, wa)
    sb.sparda_forecast_select(shape, layer.ck, f.cuda(), seq, B, idx_d[0], cnt_d[0], ws)
    sb.sparda_sparse_decode_attn(shape, layer, q_d[2], idx_d[0], cnt_d[0], seq, B, out1, wa)
    torch.cuda.synchronize()
    idx3, cnt3 = idx_d[0].cpu(), cnt_d[0].cpu()
    o1, o2 = to64(out1), to64(out2)
    for b, T in enumerate(T_list):
        for g in range(2):
            _, S = O.forecast_select_one(to64(K[b, g]), to64(f[b, g]), T, k, return_scores=True)
            check_selection(idx3[b, g], cnt3[b, g], S, T, k)
            sel3 = [int(x) for x in idx3[b, g, :int(cnt3[b, g])]]
            ref3 = O.block_sparse_attention(to64(qs[2][b, 16 * g:16 * g + 16]), to64(K[b, g]),
                                            to64(V[b, g]), sel3, T)
            check_attention(o1[b, 16 * g:16 * g + 16], ref3)
            ref2 = O.block_sparse_attention(to64(qs[1][b, 16 * g:16 * g + 16]), to64(K[b, g]),
                                            to64(V[b, g]), sels[1][b, g], T)
            check_attention(o2[b, 16 * g:16 * g + 16], ref2)
    _no_device_error(sb)


def test_attention_all_blocks_equals_dense(sb):
    T, max_ctx = 1000, 1024
    shape = sb.Shape(max_ctx=max_ctx, max_batch=1, topk=62)
    K = synth.normal_bf16((1, 2, max_ctx, 128), 51, 0)
    V = synth.normal_bf16((1, 2, max_ctx, 128), 52, 0)
    q = synth.normal_bf16((1, 32, 128), 53, 0)
    layer = sb.LayerKV.empty(shape)
    layer.k.copy_(K.cuda())
    layer.v.copy_(V.cuda())
    nb = (T - 1) // 64 + 1
    idx = torch.full((1, 2, 64), -1, dtype=torch.int32)
    idx[:, :, :nb] = torch.arange(nb, dtype=torch.int32)
    cnt = torch.full((1, 2), nb, dtype=torch.int32)
    out = torch.empty((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    ws = sb.workspace(shape, 1, sb.WS_ATTN)
    sb.sparda_sparse_decode_attn(shape, layer, q.cuda(), idx.cuda(), cnt.cuda(),
                                 torch.tensor([T], dtype=torch.int32, device="cuda"), 1, out, ws)
    torch.cuda.synchronize()
    for g in range(2):
        ref = O.dense_causal_attention(to64(q[0, 16 * g:16 * g + 16]), to64(K[0, g]), to64(V[0, g]), T)
        check_attention(to64(out[0, 16 * g:16 * g + 16]), ref)
    _no_device_error(sb)


def test_bad_seq_len_and_index_set_device_error(sb):
    shape = sb.Shape(max_ctx=1024, max_batch=2, topk=8)
    layer = sb.LayerKV.empty(shape)
    layer.k.zero_()
    layer.v.zero_()
    seq = torch.tensor([0, 5000], dtype=torch.int32, device="cuda")
    idx = torch.zeros((2, 2, 10), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((2, 2), dtype=torch.int32, device="cuda")
    ws = sb.workspace(shape, 2, sb.WS_SELECT)
    f = torch.zeros((2, 2, 128), dtype=torch.bfloat16, device="cuda")
    sb.sparda_forecast_select(shape, layer.ck, f, seq, 2, idx, cnt, ws)
    # the stream-ordered read sees the bit and clears it; the blocking read then finds it clear
    flag = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    sb.sparda_get_device_status(flag, clear=True)
    torch.cuda.synchronize()
    assert flag.item() & sb.DEV_BAD_SEQ_LEN
    assert sb.sparda_device_error(clear=True) == 0
    host_flag = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    sb.sparda_get_device_status(host_flag, clear=False)
    torch.cuda.synchronize()
    assert host_flag.item() == 0
    sb.sparda_forecast_select(shape, layer.ck, f, seq, 2, idx, cnt, ws)
    assert sb.sparda_device_error(clear=True) & sb.DEV_BAD_SEQ_LEN
    assert cnt.abs().sum().item() == 0 and (idx == -1).all()
    # a block index beyond the sequence is skipped and reported, never dereferenced
    seq = torch.tensor([100, 100], dtype=torch.int32, device="cuda")
    idx = torch.tensor([[[0, 5] + [-1] * 8] * 2] * 2, dtype=torch.int32, device="cuda")
    cnt = torch.full((2, 2), 2, dtype=torch.int32, device="cuda")
    out = torch.empty((2, 32, 128), dtype=torch.bfloat16, device="cuda")
    wa = sb.workspace(shape, 2, sb.WS_ATTN)
    q = torch.zeros((2, 32, 128), dtype=torch.bfloat16, device="cuda")
    sb.sparda_sparse_decode_attn(shape, layer, q, idx, cnt, seq, 2, out, wa)
    assert sb.sparda_device_error(clear=True) & sb.DEV_BAD_INDEX


# ------------------------------------------------------------------ baseline multi-head selector
def _mh_case(sb, K, q, T_list, k, max_ctx):
    B = len(T_list)
    shape = sb.Shape(max_ctx=max_ctx, max_batch=B, topk=k)
    ck = torch.zeros((B, 2, shape.w_cap, 128), dtype=torch.bfloat16)
    Sref = {}
    for b, T in enumerate(T_list):
        for g in range(2):
            W = O.num_windows(T - 1)
            c = O.compress_keys(to64(K[b, g]), W)
            ck[b, g, :W] = torch.from_numpy(c).to(torch.bfloat16)
            s = O.multihead_scores(to64(q[b, 16 * g:16 * g + 16]), c) if W else np.zeros(0)
            Sref[b, g] = O.pool_to_blocks(s, (T - 1) // 64 + 1)
    seq = torch.tensor(T_list, dtype=torch.int32, device="cuda")
    idx = torch.full((B, 2, k + 2), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, 2), -7, dtype=torch.int32, device="cuda")
    ws = sb.workspace(shape, B, sb.WS_MULTIHEAD)
    for rep in range(2):
        sb.sparda_multihead_select(shape, ck.cuda(), q.cuda(), seq, B, idx, cnt, ws)
        torch.cuda.synchronize()
        for b, T in enumerate(T_list):
            for g in range(2):
                check_selection(idx[b, g].cpu().numpy(), cnt[b, g].item(), Sref[b, g], T, k)
    _no_device_error(sb)
    return idx.cpu(), cnt.cpu()


@pytest.mark.parametrize("T_list,k,max_ctx", [
    ([4096], 8, 4096),
    ([1, 65, 3000, 4097], 8, 8192),
    ([8192, 5001], 32, 8192),
])
def test_multihead_select(sb, T_list, k, max_ctx):
    B = len(T_list)
    K = synth.normal_bf16((B, 2, max_ctx, 128), 91, B, k)
    q = synth.normal_bf16((B, 32, 128), 92, B, k)
    _mh_case(sb, K, q, T_list, k, max_ctx)


def test_multihead_with_identical_queries_selects_like_the_forecast(sb):
    # 16 heads all carrying the forecast vector: the summed per-head softmax is a monotone map
    # of the single-head score, so both selectors pick the same blocks
    T_list, k, max_ctx = [4096, 3001], 8, 4096
    B = len(T_list)
    case = [synth.tiny_case(s) for s in (5, 6)]
    K = torch.stack([c["K"][0] for c in case])
    f = torch.stack([c["f"][0] for c in case])
    q = f.repeat_interleave(16, dim=1)                       # [B, 32, 128]
    idx, cnt = _mh_case(sb, K, q, T_list, k, max_ctx)
    for b, T in enumerate(T_list):
        for g in range(2):
            _, S1 = O.forecast_select_one(to64(K[b, g]), to64(f[b, g]), T, k, return_scores=True)
            check_selection(idx[b, g].numpy(), cnt[b, g].item(), S1, T, k)


# ------------------------------------------------------------------ decode prologue
def test_decode_prologue_equals_its_three_calls(sb):
    # the top-k of block scores, the append and the forecast projection in one launch give
    # exactly what the selector, sparda_append_kv and sparda_forecast_project give
    T_list, k, max_ctx, hidden = [4096, 3001, 130, 2049], 8, 4096, 512
    B = len(T_list)
    shape = sb.Shape(max_ctx=max_ctx, max_batch=B, topk=k)
    K = synth.normal_bf16((B, 2, max_ctx, 128), 71, 0)
    V = synth.normal_bf16((B, 2, max_ctx, 128), 71, 1)
    f = synth.normal_bf16((B, 2, 128), 71, 2).cuda()
    kn = synth.normal_bf16((B, 2, 128), 71, 3).cuda()
    vn = synth.normal_bf16((B, 2, 128), 71, 4).cuda()
    W = synth.normal_bf16((256, hidden), 71, 5, std=0.02).cuda()
    h = synth.normal_bf16((B, hidden), 71, 6).cuda()
    seq = torch.tensor(T_list, dtype=torch.int32, device="cuda")

    def fresh():
        layer = sb.LayerKV.empty(shape)
        layer.k.copy_(K.cuda())
        layer.v.copy_(V.cuda())
        sb.sparda_compress_keys(shape, layer, seq - 1, B)
        return layer

    def slots():
        return (torch.full((B, 2, k + 2), -9, dtype=torch.int32, device="cuda"),
                torch.full((B, 2), -9, dtype=torch.int32, device="cuda"))

    la, lb = fresh(), fresh()
    ws = sb.workspace(shape, B, sb.WS_SELECT)
    idx_a, cnt_a = slots()
    sb.sparda_forecast_select(shape, la.ck, f, seq, B, idx_a, cnt_a, ws)   # leaves the block scores in ws
    sb.sparda_append_kv(shape, la, kn, vn, seq, B)
    f_a = torch.empty((B, 256), dtype=torch.bfloat16, device="cuda")
    sb.sparda_forecast_project(W, h, f_a)
    idx_b, cnt_b = slots()
    f_b = torch.empty((B, 256), dtype=torch.bfloat16, device="cuda")
    sb.sparda_decode_prologue(shape, lb, kn, vn, seq, B, ws_scores=ws, idx=idx_b, cnt=cnt_b, W_next=W, h=h,
                              forecast_next=f_b)
    torch.cuda.synchronize()
    assert torch.equal(idx_a, idx_b) and torch.equal(cnt_a, cnt_b)
    assert torch.equal(f_a, f_b)
    assert torch.equal(la.k, lb.k) and torch.equal(la.v, lb.v) and torch.equal(la.ck, lb.ck)
    # the append alone (no scores, no projection) leaves the selection untouched
    idx_c, cnt_c = slots()
    sb.sparda_decode_prologue(shape, fresh(), kn, vn, seq, B, idx=idx_c, cnt=cnt_c)
    torch.cuda.synchronize()
    assert (idx_c == -9).all() and (cnt_c == -9).all()
    _no_device_error(sb)


@pytest.mark.parametrize("B", [3, 18])
def test_score_then_prologue_top_k_equals_select(sb, B):
    # sparda_forecast_score leaves the block scores that sparda_decode_prologue's top-k turns
    # into exactly the selection sparda_forecast_select makes; B = 3 takes the queue-fed
    # scoring (6 sequence-groups), B = 18 the fixed ranges (36)
    k, max_ctx = 8, 4096
    T_list = [max_ctx - 7 * b for b in range(B)]
    shape = sb.Shape(max_ctx=max_ctx, max_batch=B, topk=k)
    K = synth.normal_bf16((B, 2, max_ctx, 128), 73, B)
    f = synth.normal_bf16((B, 2, 128), 74, B).cuda()
    seq = torch.tensor(T_list, dtype=torch.int32, device="cuda")
    layer = sb.LayerKV.empty(shape)
    layer.k.copy_(K.cuda())
    sb.sparda_compress_keys(shape, layer, seq - 1, B)
    idx_a = torch.full((B, 2, k + 2), -9, dtype=torch.int32, device="cuda")
    cnt_a = torch.full((B, 2), -9, dtype=torch.int32, device="cuda")
    idx_b, cnt_b = idx_a.clone(), cnt_a.clone()
    ws_a = sb.workspace(shape, B, sb.WS_SELECT)
    ws_b = sb.workspace(shape, B, sb.WS_SELECT)
    sb.sparda_forecast_select(shape, layer.ck, f, seq, B, idx_a, cnt_a, ws_a)
    kn = torch.zeros((B, 2, 128), dtype=torch.bfloat16, device="cuda")
    for rep in range(2):                                  # the workspace is reusable as left
        sb.sparda_forecast_score(shape, layer.ck, f, seq, B, ws_b)
        sb.sparda_decode_prologue(shape, sb.LayerKV.empty(shape), kn, kn, seq, B, ws_scores=ws_b, idx=idx_b,
                                  cnt=cnt_b)
        torch.cuda.synchronize()
        assert torch.equal(idx_a, idx_b) and torch.equal(cnt_a, cnt_b)
    _no_device_error(sb)


def _planted_scores(kind, nb, rng):
    S = rng.standard_normal(nb).astype(np.float32)
    if kind == "signed_zeros":          # -0 and +0 are equal scores: ties go to the lower block
        S = np.where(rng.random(nb) < 0.5, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
        S[rng.choice(nb, 5, replace=False)] = 1.0
        S[rng.choice(nb, 5, replace=False)] = -1.0
    elif kind == "plateau":             # more equal maxima than the fast path lists
        S -= 10.0
        S[rng.choice(nb, nb * 3 // 4, replace=False)] = 3.0
    elif kind == "few_distinct":        # heavy ties at every level
        S = rng.integers(0, 4, nb).astype(np.float32)
    elif kind == "one_warp_high":       # every high score in the lanes of one top-k warp
        S[np.arange(nb) % 256 < 32] += 100.0
    elif kind == "infinities":          # non-finite scores rank above / below every finite one
        S[rng.choice(nb, 3, replace=False)] = np.inf
        S[rng.choice(nb, 40, replace=False)] = -np.inf
    return S


@pytest.mark.parametrize("kind", ["normal", "signed_zeros", "plateau", "few_distinct", "one_warp_high",
                                  "infinities"])
@pytest.mark.parametrize("k,max_ctx", [(32, 131072), (62, 262144), (8, 8192)])
def test_prologue_top_k_of_planted_scores(sb, kind, k, max_ctx):
    # block scores written straight into the selection workspace: the prologue's top-k must
    # give exactly the oracle's selection (block 0, the tail block and the k best others, ties
    # to the lower block) for each (sequence, group) row, whatever the score distribution
    nb = max_ctx // 64
    T_list = [max_ctx, max_ctx - 100 * 64 + 5, 300 * 64 + 1 if max_ctx > 300 * 64 else 40 * 64, 3 * 64, 33 * 64 + 1]
    B = len(T_list)
    shape = sb.Shape(max_ctx=max_ctx, max_batch=B, topk=k)
    G = shape.n_groups
    rng = np.random.default_rng([5, k, nb, len(kind)])
    S = np.stack([_planted_scores(kind, nb, rng) for _ in range(B * G)])
    ws = sb.workspace(shape, B, sb.WS_SELECT)
    off = sb.sparda_block_scores_offset(shape)
    ws[off:off + S.nbytes].view(torch.float32).view(B * G, nb).copy_(torch.from_numpy(S))
    seq = torch.tensor(T_list, dtype=torch.int32, device="cuda")
    kn = torch.zeros((B, G, 128), dtype=torch.bfloat16, device="cuda")
    idx = torch.full((B, G, k + 2), -9, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, G), -9, dtype=torch.int32, device="cuda")
    sb.sparda_decode_prologue(shape, sb.LayerKV.empty(shape), kn, kn, seq, B, ws_scores=ws, idx=idx, cnt=cnt)
    torch.cuda.synchronize()
    idx, cnt = idx.cpu(), cnt.cpu()
    for b, T in enumerate(T_list):
        for g in range(G):
            want = O.select_blocks(S[b * G + g].astype(np.float64), T, k)
            got = idx[b, g].tolist()
            assert cnt[b, g].item() == len(want), (kind, b, g)
            assert got == want + [-1] * (k + 2 - len(want)), (kind, b, g)
    _no_device_error(sb)


def test_append_window_means_round_exactly(sb):
    # The window that token 31 completes, built so that the exact means hit the cases that a
    # slip in the append's exact summation and rounding would get wrong: halfway cases that
    # round down or up to even, means of mixed signs and magnitudes, all-zero and negative
    # zero windows, keys below 2^-40 and of 2^11 or more (summed another way), sums that
    # carry into the next binade. Compared bit for bit with the oracle's compressed key.
    T = 32
    K = synth.normal_bf16((1, 2, 256, 128), 81, 0).double().numpy()
    W = np.zeros((32, 128))
    cases = [
        {0: 32.0, 1: 0.125},                  # mean 1 + 2^-8: halfway, rounds down to even 1.0
        {0: 32.0, 1: 0.25, 2: 0.125},         # mean 1 + 3*2^-8: halfway, rounds up to 1 + 2^-6
        {0: -32.0, 1: -0.125},                # negative halfway
        {0: 32.0, 1: 0.125, 2: 2.0 ** -30},   # just above halfway: rounds up
        {0: 63.75, 1: 0.125, 2: 0.0625},      # mean 2 - 2^-9 rounds up to 2.0: carries into the exponent
        {0: 4096.0, 1: 1.0},                  # a key of 2^12: the float64 path
        {0: 3008.0, 1: -2992.0, 2: 0.5},      # large cancelling keys: the float64 path
        {0: 2.0 ** -41, 1: 2.0 ** -20},       # a key below 2^-40: the float64 path
        {0: 2.0 ** -40, 1: 2.0 ** -33},       # the smallest magnitudes the integer path takes
        {0: 1.0, 1: -1.0},                    # exact zero
    ]
    for d, c in enumerate(cases):
        for r, x in c.items():
            W[r, d] = x
    W[:, len(cases)] = -0.0                   # a window of negative zeros
    W[:, len(cases) + 1:] = K[0, 0, :32, len(cases) + 1:]
    Kw = torch.from_numpy(W).to(torch.bfloat16)
    assert torch.equal(Kw.double(), torch.from_numpy(W)), "the crafted keys must be bf16 values"
    shape = sb.Shape(max_ctx=256, max_batch=1, topk=8)
    layer = sb.LayerKV.empty(shape)
    layer.k.zero_()
    layer.v.zero_()
    for g in range(2):
        layer.k[0, g, :31] = Kw[:31].cuda()
    seq = torch.tensor([T], dtype=torch.int32, device="cuda")
    kn = torch.stack([Kw[31], Kw[31]]).view(1, 2, 128).cuda()
    sb.sparda_append_kv(shape, layer, kn, kn, seq, 1)
    torch.cuda.synchronize()
    got = layer.ck[0, :, 0].cpu().view(torch.int16)
    want = torch.from_numpy(O.compress_keys(Kw.double().numpy(), 1)[0]).to(torch.bfloat16).view(torch.int16)
    for g in range(2):
        assert torch.equal(got[g], want), (g, (got[g] != want).nonzero())
    _no_device_error(sb)


@pytest.mark.parametrize("nbytes", [16, 4096 + 16, 1 << 20, (64 << 20) + 48])
def test_copy_between_device_and_pinned_host(sb, nbytes):
    # sparda_copy: device to device, pinned host to device, device to pinned host; sizes from
    # one 16-byte word to more words than one pass of the grid covers
    n = nbytes // 2
    g = torch.Generator().manual_seed(nbytes)
    src_host = torch.randint(-30000, 30000, (n,), dtype=torch.int16, generator=g).pin_memory()
    dev = torch.empty(n, dtype=torch.int16, device="cuda")
    sb.sparda_copy(dev, src_host)
    dev2 = torch.empty_like(dev)
    sb.sparda_copy(dev2, dev)
    back = torch.zeros(n, dtype=torch.int16).pin_memory()
    sb.sparda_copy(back, dev2)
    torch.cuda.synchronize()
    assert torch.equal(back, src_host)
    assert torch.equal(dev2.cpu(), src_host)


def test_copy_rejects_pageable_host_memory(sb):
    dev = torch.empty(64, dtype=torch.int16, device="cuda")
    with pytest.raises(sb.SpardaError):
        sb.sparda_copy(dev, torch.zeros(64, dtype=torch.int16))          # not pinned
