"""Host-side checks of the C ABI: the library loads without a GPU, exports every function
include/sparda.h declares, and rejects bad arguments before launching anything."""
import ctypes

import pytest

from block_sparse_attention_forecast_gb300 import build as _build

_build.build()

import block_sparse_attention_forecast_gb300.binding as sb  # noqa: E402


def test_library_exports_every_declared_function():
    names = sb.header_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(sb.lib, n), n
        assert hasattr(sb, n), "binding lacks " + n


def test_status_strings_and_version():
    assert sb.sparda_abi_version() == 1
    assert sb.status_string(sb.OK) == "ok"
    assert "workspace" in sb.status_string(sb.ERR_WORKSPACE_TOO_SMALL)
    assert sb.status_string(12345) == "unknown status"


def test_shape_checks():
    assert sb.sparda_check_shape(sb.Shape()) == sb.OK
    for bad in (dict(head_dim=64), dict(heads_per_group=8), dict(block=128), dict(win_kernel=16),
                dict(topk=0), dict(topk=63), dict(max_ctx=100), dict(max_ctx=524288),
                dict(n_groups=0), dict(max_batch=0), dict(max_batch=4096, n_groups=8, max_ctx=262144)):
        assert sb.sparda_check_shape(sb.Shape(**bad)) == sb.ERR_UNSUPPORTED_SHAPE, bad
    assert sb.lib.sparda_check_shape(None) == sb.ERR_INVALID_ARG


def test_workspace_sizes():
    s = sb.Shape(n_groups=2, topk=32, max_ctx=131072 + 64, max_batch=16)
    nb = s.max_ctx // 64
    sel = sb.sparda_workspace_bytes(s, 16, sb.WS_SELECT)
    assert sel >= 16 * 2 * 4 + 16 * 2 * nb * 4
    att = sb.sparda_workspace_bytes(s, 16, sb.WS_ATTN)
    assert att >= 16 * 2 * 17 * 16 * 128 * 4
    assert sb.sparda_workspace_bytes(s, 0, sb.WS_SELECT) == 0
    assert sb.sparda_workspace_bytes(s, 17, sb.WS_SELECT) == 0
    assert sb.sparda_workspace_bytes(s, 4, 99) == 0
    # the block scores fill the end of the selection workspace, after its counters
    off = sb.sparda_block_scores_offset(s)
    assert off % 16 == 0 and 16 * 2 * 4 <= off and off + 16 * 2 * nb * 4 <= sel
    assert sb.sparda_block_scores_offset(sb.Shape(max_ctx=100)) == 0
    assert sb.sparda_prefetch_default_ctas(31) == 64 and sb.sparda_prefetch_default_ctas(32) == 152


def test_bad_arguments_are_rejected_before_any_launch():
    s = sb.Shape(max_batch=2, max_ctx=4096)
    sh = ctypes.byref(s.c())
    P = ctypes.c_void_p
    fake = P(1 << 20)          # never dereferenced: the checks fail first
    odd = P((1 << 20) + 8)     # not 16-byte aligned
    assert sb.lib.sparda_forecast_select(sh, None, fake, fake, 1, fake, fake, fake, 1 << 20, None) == sb.ERR_INVALID_ARG
    assert sb.lib.sparda_forecast_select(sh, odd, fake, fake, 1, fake, fake, fake, 1 << 20, None) == sb.ERR_MISALIGNED
    assert sb.lib.sparda_forecast_select(sh, fake, fake, fake, 3, fake, fake, fake, 1 << 20, None) == sb.ERR_INVALID_ARG
    assert sb.lib.sparda_forecast_select(sh, fake, fake, fake, 1, fake, fake, fake, 16, None) == sb.ERR_WORKSPACE_TOO_SMALL
    layer = sb.c_layer_kv(None, None, None, None, None, 0, 0)
    assert sb.lib.sparda_append_kv(sh, ctypes.byref(layer), fake, fake, fake, 1, None) == sb.ERR_INVALID_ARG
    assert sb.lib.sparda_sparse_decode_attn(sh, ctypes.byref(layer), None, None, None, fake, fake, fake, 1, fake, fake, 1 << 30, None) == sb.ERR_INVALID_ARG
    assert sb.lib.sparda_forecast_project(fake, fake, 12, 4096, 1, fake, None) == sb.ERR_UNSUPPORTED_SHAPE
    assert sb.lib.sparda_forecast_project(odd, fake, 256, 4096, 1, fake, None) == sb.ERR_MISALIGNED
    resident = sb.c_layer_kv(1 << 20, 1 << 20, 1 << 20, None, None, 0, 0)
    assert sb.lib.sparda_prefetch_blocks(sh, ctypes.byref(resident), fake, fake, fake, 1, fake, fake, 0, None) == sb.ERR_INVALID_ARG
    offl = sb.c_layer_kv(1 << 20, 1 << 20, 1 << 20, None, None, 1, 0)
    assert sb.lib.sparda_prefetch_blocks(sh, ctypes.byref(offl), fake, fake, fake, 1, fake, fake, 0, None) == sb.ERR_INVALID_ARG
    assert sb.lib.sparda_prefetch_blocks(sh, ctypes.byref(resident), fake, fake, fake, 1, fake, fake, -1, None) == sb.ERR_INVALID_ARG
    assert sb.lib.sparda_forecast_score(sh, None, fake, fake, 1, fake, 1 << 20, None) == sb.ERR_INVALID_ARG
    assert sb.lib.sparda_forecast_score(sh, odd, fake, fake, 1, fake, 1 << 20, None) == sb.ERR_MISALIGNED
    assert sb.lib.sparda_forecast_score(sh, fake, fake, fake, 1, fake, 16, None) == sb.ERR_WORKSPACE_TOO_SMALL
    assert sb.lib.sparda_copy(None, fake, 256, None) == sb.ERR_INVALID_ARG
    assert sb.lib.sparda_copy(fake, fake, 0, None) == sb.ERR_INVALID_ARG
    assert sb.lib.sparda_copy(fake, fake, 100, None) == sb.ERR_INVALID_ARG            # not a multiple of 16
    assert sb.lib.sparda_copy(odd, fake, 256, None) == sb.ERR_MISALIGNED
    assert sb.lib.sparda_copy(fake, odd, 256, None) == sb.ERR_MISALIGNED


def test_pipelined_entries_reject_bad_arguments():
    s = sb.Shape(max_batch=2, max_ctx=4096)
    sh = ctypes.byref(s.c())
    P = ctypes.c_void_p
    fake = P(1 << 20)
    odd = P((1 << 20) + 8)
    resident = sb.c_layer_kv(1 << 20, 1 << 20, 1 << 20, None, None, 0, 0)
    L = ctypes.byref(resident)
    prologue = sb.lib.sparda_decode_prologue
    # block scores to select from, but nowhere to write the selection
    assert prologue(sh, L, fake, fake, fake, 1 << 24, None, None, None, None, 0, None, fake, 1, None) == sb.ERR_INVALID_ARG
    # a score workspace too small for the batch
    assert prologue(sh, L, fake, fake, fake, 16, fake, fake, None, None, 0, None, fake, 1, None) == sb.ERR_WORKSPACE_TOO_SMALL
    # a projection whose hidden size is not a multiple of 32, or without its input
    assert prologue(sh, L, fake, fake, None, 0, None, None, fake, fake, 100, fake, fake, 1, None) == sb.ERR_UNSUPPORTED_SHAPE
    assert prologue(sh, L, fake, fake, None, 0, None, None, fake, None, 4096, fake, fake, 1, None) == sb.ERR_INVALID_ARG
    assert prologue(sh, L, odd, fake, None, 0, None, None, None, None, 0, None, fake, 1, None) == sb.ERR_MISALIGNED
    assert prologue(sh, L, fake, fake, None, 0, None, None, None, None, 0, None, fake, 3, None) == sb.ERR_INVALID_ARG
    # the score workspace may not be the attention workspace
    score = sb.lib.sparda_attend_and_score
    assert score(sh, L, None, None, fake, fake, fake, fake, fake, 1 << 30, fake, fake, fake, 1 << 30, None, 0, fake,
                 1, None) == sb.ERR_INVALID_ARG
    # the L2 hint must be 16-byte aligned and a whole number of 16-byte granules
    assert score(sh, L, None, None, fake, fake, fake, fake, fake, 1 << 30, fake, fake, P(1 << 22), 1 << 30, odd, 4096,
                 fake, 1, None) == sb.ERR_MISALIGNED
    assert score(sh, L, None, None, fake, fake, fake, fake, fake, 1 << 30, fake, fake, P(1 << 22), 1 << 30, fake, 100,
                 fake, 1, None) == sb.ERR_MISALIGNED

