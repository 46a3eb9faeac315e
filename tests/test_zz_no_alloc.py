"""The allocation-free selector entry point (sparda_forecast_select_static).

It exists for callers that cannot allocate device memory -- a plugin that its host engine
hands only input and output tensors, or a serving loop that must not allocate once it runs --
so its scratch is a fixed array inside the library. These tests check that it returns
exactly what the workspace-taking sparda_forecast_select returns, on two calls in a row (the
shared array keeps the previous call's contents, which must not leak into the next result),
and that requests larger than its fixed scratch are refused before anything is launched.
The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import synth

from block_sparse_attention_forecast_gb300 import build as _build

_build.build()

import block_sparse_attention_forecast_gb300.binding as sb  # noqa: E402


def _static_status(shape, batch):
    fake = ctypes.c_void_p(1 << 20)         # aligned, never dereferenced: the size check comes first
    return sb.lib.sparda_forecast_select_static(ctypes.byref(shape.c()), fake, fake, fake, batch, fake, fake,
                                                None)


def test_oversized_request_is_refused_without_launch():
    # 64 sequences x 8 groups x 4096 blocks of float scores need 8 MiB, more than the 4 MiB scratch
    shape = sb.Shape(n_groups=8, topk=32, max_ctx=262144, max_batch=64)
    st = _static_status(shape, 64)
    assert st == sb.ERR_STATIC_SCRATCH_LIMIT
    assert "allocation-free" in sb.status_string(st)


# At 2 groups and context 131072 a sequence takes 2 x 2048 block scores of 4 bytes (16 KiB);
# beside the 16 KiB of counters, 255 sequences fill the 4 MiB scratch exactly.
LIMIT_BATCH_128K = 255


def test_size_limit_is_exact():
    assert 4 * 4096 + 4 * LIMIT_BATCH_128K * 2 * (131072 // 64) == 4 << 20
    shape = sb.Shape(n_groups=2, topk=32, max_ctx=131072, max_batch=LIMIT_BATCH_128K + 1)
    assert _static_status(shape, LIMIT_BATCH_128K + 1) == sb.ERR_STATIC_SCRATCH_LIMIT
    assert _static_status(sb.Shape(n_groups=4097, topk=8, max_ctx=64, max_batch=1), 1) == sb.ERR_STATIC_SCRATCH_LIMIT


@pytest.mark.gpu
def test_static_select_matches_workspace_select_twice(cuda_ok):
    sb.sparda_device_error(clear=True)
    T_list, k, max_ctx = [4096, 3000, 65, 2500], 8, 4096
    B = len(T_list)
    shape = sb.Shape(n_groups=2, topk=k, max_ctx=max_ctx, max_batch=B)
    layer = sb.LayerKV.empty(shape)
    layer.k.copy_(synth.normal_bf16((B, 2, max_ctx, 128), 61, 0).cuda())
    layer.v.zero_()
    seq_prev = torch.tensor([t - 1 for t in T_list], dtype=torch.int32, device="cuda")
    sb.sparda_compress_keys(shape, layer, seq_prev, B)
    seq = torch.tensor(T_list, dtype=torch.int32, device="cuda")
    ws = sb.workspace(shape, B, sb.WS_SELECT)
    for call in range(2):
        f = synth.normal_bf16((B, 2, 128), 62, call).cuda()    # a different forecast each call
        idx_ref = torch.full((B, 2, k + 2), -9, dtype=torch.int32, device="cuda")
        cnt_ref = torch.full((B, 2), -9, dtype=torch.int32, device="cuda")
        sb.sparda_forecast_select(shape, layer.ck, f, seq, B, idx_ref, cnt_ref, ws)
        idx = torch.full((B, 2, k + 2), -9, dtype=torch.int32, device="cuda")
        cnt = torch.full((B, 2), -9, dtype=torch.int32, device="cuda")
        sb.sparda_forecast_select_static(shape, layer.ck, f, seq, B, idx, cnt)
        torch.cuda.synchronize()
        # block indices are integers: the tolerance the other selector tests use is exact
        assert torch.equal(idx, idx_ref), (call, idx, idx_ref)
        assert torch.equal(cnt, cnt_ref), (call, cnt, cnt_ref)
    assert sb.sparda_device_error(clear=True) == 0


@pytest.mark.gpu
@pytest.mark.parametrize("B", [64, LIMIT_BATCH_128K])
def test_static_select_at_context_131072(cuda_ok, B):
    """The documented example size (batch 64, 2 groups, context 131072) and the largest batch
    that fits the scratch at that context, each against sparda_forecast_select."""
    sb.sparda_device_error(clear=True)
    T, k = 131072, 32
    shape = sb.Shape(n_groups=2, topk=k, max_ctx=T, max_batch=B)
    ck = synth.normal_bf16_device((B, 2, shape.w_cap, 128), 63, "cuda", std=0.18)
    seq = torch.full((B,), T, dtype=torch.int32, device="cuda")
    seq[1] = T - 1000                       # one shorter sequence
    ws = sb.workspace(shape, B, sb.WS_SELECT)
    for call in range(2):
        f = synth.normal_bf16_device((B, 2, 128), 64 + call, "cuda")
        idx_ref = torch.full((B, 2, k + 2), -9, dtype=torch.int32, device="cuda")
        cnt_ref = torch.full((B, 2), -9, dtype=torch.int32, device="cuda")
        sb.sparda_forecast_select(shape, ck, f, seq, B, idx_ref, cnt_ref, ws)
        idx = torch.full((B, 2, k + 2), -9, dtype=torch.int32, device="cuda")
        cnt = torch.full((B, 2), -9, dtype=torch.int32, device="cuda")
        sb.sparda_forecast_select_static(shape, ck, f, seq, B, idx, cnt)
        torch.cuda.synchronize()
        assert torch.equal(idx, idx_ref), call
        assert torch.equal(cnt, cnt_ref), call
        assert (cnt == k + 2).all()
    assert sb.sparda_device_error(clear=True) == 0
    del ck, ws
    torch.cuda.empty_cache()
