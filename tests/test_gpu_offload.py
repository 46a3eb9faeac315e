"""The host-offload path: the UVA gather of selected blocks from pinned host memory into
staging, appends into the hot ring (with the flush of a filled block to the host cache), and
attention that reads staging and the hot ring -- against the fp64 oracle."""
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


def _offloaded_layer(sb, shape, K, V, n_cached):
    layer = sb.LayerKV.empty(shape, on_host=True)
    layer.k.copy_(K)
    layer.v.copy_(V)
    sb.fill_hot_from_host(layer, n_cached)
    seq = torch.tensor(n_cached, dtype=torch.int32, device="cuda")
    sb.sparda_compress_keys(shape, layer, seq, len(n_cached))
    return layer


@pytest.mark.parametrize("T_list,k,n_ctas", [([3000, 2001], 8, 0), ([4096, 130, 65], 8, 3), ([2600, 4000], 32, 16)])
def test_gather_and_attention_from_staging(sb, T_list, k, n_ctas):
    B, max_ctx = len(T_list), 4096
    shape = sb.Shape(topk=k, max_ctx=max_ctx, max_batch=B)
    K = synth.normal_bf16((B, 2, max_ctx, 128), 71, B)
    V = synth.normal_bf16((B, 2, max_ctx, 128), 72, B)
    layer = _offloaded_layer(sb, shape, K, V, [t - 1 for t in T_list])
    f = synth.normal_bf16((B, 2, 128), 73, B)
    q = synth.normal_bf16((B, 32, 128), 74, B)
    kn = synth.normal_bf16((B, 2, 128), 75, B)
    vn = synth.normal_bf16((B, 2, 128), 76, B)
    seq = torch.tensor(T_list, dtype=torch.int32, device="cuda")
    idx = torch.zeros((B, 2, k + 2), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B, 2), dtype=torch.int32, device="cuda")
    sb.sparda_forecast_select(shape, layer.ck, f.cuda(), seq, B, idx, cnt, sb.workspace(shape, B, sb.WS_SELECT))
    st = (B, 2, k + 2, 64, 128)
    sk = torch.zeros(st, dtype=torch.bfloat16, device="cuda")
    sv = torch.zeros(st, dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    sb.sparda_prefetch_blocks(shape, layer, idx, cnt, seq, B, sk, sv, n_ctas=n_ctas, stream=side)
    sb.sparda_append_kv(shape, layer, kn.cuda(), vn.cuda(), seq, B)
    torch.cuda.current_stream().wait_stream(side)
    out = torch.zeros((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    sb.sparda_sparse_decode_attn(shape, layer, q.cuda(), idx, cnt, seq, B, out, sb.workspace(shape, B, sb.WS_ATTN),
                                 staging_k=sk, staging_v=sv)
    torch.cuda.synchronize()
    Kd, Vd = to64(K), to64(V)
    idx_h, cnt_h, o = idx.cpu().numpy(), cnt.cpu().numpy(), to64(out)
    for b, T in enumerate(T_list):
        Kd[b, :, T - 1] = to64(kn[b])
        Vd[b, :, T - 1] = to64(vn[b])
        tb = (T - 1) // 64
        for g in range(2):
            # compressed keys built from host + hot ring match the oracle bit for bit
            W = O.num_windows(T - 1)
            assert np.array_equal(to64(layer.ck[b, g, :W]), O.compress_keys(to64(K[b, g]), W))
            sel, S = O.forecast_select_one(Kd[b, g], to64(f[b, g]), T, k, return_scores=True)
            check_selection(idx_h[b, g], cnt_h[b, g], S, T, k)
            gsel = list(idx_h[b, g, :cnt_h[b, g]])
            # the gather copied exactly the host blocks of the scored slots
            for s, j in enumerate(gsel):
                if j in (0, tb):
                    continue
                assert torch.equal(sk[b, g, s].cpu(), K[b, g, j * 64:(j + 1) * 64]), (b, g, s, j)
                assert torch.equal(sv[b, g, s].cpu(), V[b, g, j * 64:(j + 1) * 64]), (b, g, s, j)
            ref = O.block_sparse_attention(to64(q[b, 16 * g:16 * g + 16]), Kd[b, g], Vd[b, g], gsel, T)
            check_attention(o[b, 16 * g:16 * g + 16], ref)
    assert sb.sparda_device_error(clear=True) == 0


def test_offloaded_append_flushes_full_blocks(sb):
    B, max_ctx, n0, steps = 2, 1024, [250, 183], 12
    shape = sb.Shape(topk=8, max_ctx=max_ctx, max_batch=B)
    K = synth.normal_bf16((B, 2, max_ctx, 128), 81, 0)
    V = synth.normal_bf16((B, 2, max_ctx, 128), 82, 0)
    layer = _offloaded_layer(sb, shape, K, V, n0)
    Kd, Vd = to64(K), to64(V)
    seq = torch.zeros(B, dtype=torch.int32, device="cuda")
    for s in range(steps):
        T = [n + s + 1 for n in n0]
        kn = synth.normal_bf16((B, 2, 128), 83, s)
        vn = synth.normal_bf16((B, 2, 128), 84, s)
        seq.copy_(torch.tensor(T, dtype=torch.int32))
        sb.sparda_append_kv(shape, layer, kn.cuda(), vn.cuda(), seq, B)
        for b in range(B):
            Kd[b, :, T[b] - 1] = to64(kn[b])
            Vd[b, :, T[b] - 1] = to64(vn[b])
    torch.cuda.synchronize()
    hk, hv = to64(layer.hot_k), to64(layer.hot_v)
    for b in range(B):
        n = n0[b] + steps
        tb = (n - 1) // 64
        # every block completed during the steps is now in the host cache
        for j in range(n0[b] // 64, tb):
            assert np.array_equal(to64(layer.k[b, :, j * 64:(j + 1) * 64]), Kd[b, :, j * 64:(j + 1) * 64]), (b, j)
            assert np.array_equal(to64(layer.v[b, :, j * 64:(j + 1) * 64]), Vd[b, :, j * 64:(j + 1) * 64]), (b, j)
        # the tail block's rows written so far are in its hot slot
        r = n - tb * 64
        assert np.array_equal(hk[b, :, sb.hot_slot(tb), :r], Kd[b, :, tb * 64:n])
        assert np.array_equal(hv[b, :, sb.hot_slot(tb), :r], Vd[b, :, tb * 64:n])
        for g in range(2):
            W = O.num_windows(n)
            assert np.array_equal(to64(layer.ck[b, g, :W]), O.compress_keys(Kd[b, g], W)), (b, g)
    assert sb.sparda_device_error(clear=True) == 0
