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


def test_oversized_request_is_refused_without_launch():
    # 64 sequences x 8 groups x 4096 blocks of float scores need 8 MiB, more than the 4 MiB scratch
    shape = sb.Shape(n_groups=8, topk=32, max_ctx=262144, max_batch=64)
    fake = ctypes.c_void_p(1 << 20)
    st = sb.lib.sparda_forecast_select_static(ctypes.byref(shape.c()), fake, fake, fake, 64, fake, fake, None)
    assert st == sb.ERR_STATIC_SCRATCH_LIMIT
    assert "allocation-free" in sb.status_string(st)


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
