"""ctypes binding of libsparda (include/sparda.h).

Argument marshalling only: every function below takes torch tensors (or plain integers),
passes their device addresses and the current CUDA stream to the C entry point of the same
name, and raises SpardaError on a non-zero status. Every computation happens in the CUDA
kernels of libsparda. There is no fallback: if the library is missing, importing this module
fails with an error that says how to build it.
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass

import torch

__all__ = [
    "lib", "LIB_PATH", "HEADER_PATH", "SpardaError", "Shape", "LayerKV", "workspace",
    "hot_slot", "fill_hot_from_host",
    "header_functions", "status_string", "num_windows", "c_shape", "c_layer_kv",
    "sparda_abi_version", "sparda_status_string", "sparda_check_shape", "sparda_workspace_bytes",
    "sparda_block_scores_offset", "sparda_device_error", "sparda_get_device_status",
    "sparda_prefetch_default_ctas", "sparda_append_kv", "sparda_compress_keys",
    "sparda_forecast_project", "sparda_forecast_select", "sparda_sparse_decode_attn",
    "sparda_prefetch_blocks", "sparda_multihead_select", "sparda_forecast_select_static", "sparda_attend_and_select",
    "sparda_attend_and_score", "sparda_decode_prologue", "sparda_forecast_score", "sparda_copy",
    "sparda_prefill_forecast_select", "sparda_prefill_multihead_select", "sparda_prefill_attn",
    "sparda_prefetch_blocks_cached", "sparda_sparse_decode_attn_cached", "BlockCache",
    "sparda_prefetch_blocks_copy_engine",
    "OK", "ERR_INVALID_ARG", "ERR_UNSUPPORTED_SHAPE", "ERR_MISALIGNED", "ERR_NOT_MAPPED_HOST",
    "ERR_WORKSPACE_TOO_SMALL", "ERR_CUDA", "ERR_STATIC_SCRATCH_LIMIT", "DEV_WAIT_TIMEOUT", "DEV_BAD_SEQ_LEN", "DEV_BAD_INDEX",
    "WS_SELECT", "WS_ATTN", "WS_MULTIHEAD", "WS_PREFILL", "BLOCK", "WIN_KERNEL", "WIN_STRIDE",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
# SPARDA_LIB may name another build of the same library (the per-CTA timeline variant)
LIB_PATH = os.environ.get("SPARDA_LIB") or os.path.join(_PKG, "_lib", "libsparda.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "sparda.h")

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED_SHAPE = -2
ERR_MISALIGNED = -3
ERR_NOT_MAPPED_HOST = -4
ERR_WORKSPACE_TOO_SMALL = -5
ERR_CUDA = -6
ERR_STATIC_SCRATCH_LIMIT = -7

DEV_WAIT_TIMEOUT = 1
DEV_BAD_SEQ_LEN = 2
DEV_BAD_INDEX = 4

WS_SELECT = 1
WS_ATTN = 2
WS_MULTIHEAD = 3
WS_PREFILL = 4

BLOCK = 64
WIN_KERNEL = 32
WIN_STRIDE = 16


class SpardaError(RuntimeError):
    def __init__(self, name, status):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (name, status_string(status), status))


class c_shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_groups", "heads_per_group", "head_dim", "block", "win_kernel", "win_stride",
        "topk", "max_ctx", "max_batch")]


class c_layer_kv(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("ck", ctypes.c_void_p),
                ("hot_k", ctypes.c_void_p), ("hot_v", ctypes.c_void_p),
                ("on_host", ctypes.c_int32), ("reserved", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "libsparda.so is not built (%s). Build it with "
            "`python -m block_sparse_attention_forecast_gb300.build` (nvcc, CUDA 13)." % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    SH, LY = ctypes.POINTER(c_shape), ctypes.POINTER(c_layer_kv)
    sig = {
        "sparda_abi_version": (I32, []),
        "sparda_status_string": (ctypes.c_char_p, [I32]),
        "sparda_check_shape": (I32, [SH]),
        "sparda_workspace_bytes": (SZ, [SH, I32, I32]),
        "sparda_block_scores_offset": (SZ, [SH]),
        "sparda_device_error": (I32, [ctypes.POINTER(I32), I32]),
        "sparda_get_device_status": (I32, [P, I32, P]),
        "sparda_prefetch_default_ctas": (I32, [I32]),
        "sparda_append_kv": (I32, [SH, LY, P, P, P, I32, P]),
        "sparda_compress_keys": (I32, [SH, LY, P, I32, P]),
        "sparda_forecast_project": (I32, [P, P, I32, I32, I32, P, P]),
        "sparda_forecast_select": (I32, [SH, P, P, P, I32, P, P, P, SZ, P]),
        "sparda_sparse_decode_attn": (I32, [SH, LY, P, P, P, P, P, P, I32, P, P, SZ, P]),
        "sparda_prefetch_blocks": (I32, [SH, LY, P, P, P, I32, P, P, I32, P]),
        "sparda_multihead_select": (I32, [SH, P, P, P, I32, P, P, P, SZ, P]),
        "sparda_forecast_select_static": (I32, [SH, P, P, P, I32, P, P, P]),
        "sparda_attend_and_select": (I32, [SH, LY, P, P, P, P, P, P, P, SZ, P, P, P, P, P, SZ, P, I32, P]),
        "sparda_attend_and_score": (I32, [SH, LY, P, P, P, P, P, P, P, SZ, P, P, P, SZ, P, SZ, P, I32, P]),
        "sparda_decode_prologue": (I32, [SH, LY, P, P, P, SZ, P, P, P, P, I32, P, P, I32, P]),
        "sparda_copy": (I32, [P, P, SZ, P]),
        "sparda_forecast_score": (I32, [SH, P, P, P, I32, P, SZ, P]),
        "sparda_prefill_forecast_select": (I32, [SH, P, P, P, I32, P, P, P, SZ, P]),
        "sparda_prefill_multihead_select": (I32, [SH, P, P, P, I32, P, P, P, SZ, P]),
        "sparda_prefill_attn": (I32, [SH, LY, P, P, P, P, I32, P, P]),
        "sparda_prefetch_blocks_cached": (I32, [SH, LY, P, P, P, I32, P, P, P, I32, P, P, P, I32, P]),
        "sparda_prefetch_blocks_copy_engine": (I32, [SH, LY, P, P, P, I32, P, P, P, P]),
        "sparda_sparse_decode_attn_cached": (I32, [SH, LY, P, P, I32, P, P, P, P, P, I32, P, P, SZ, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def header_functions():
    """Names of the functions include/sparda.h declares."""
    with open(HEADER_PATH) as fh:
        text = fh.read()
    return sorted(set(re.findall(r"^\s*(?:int32_t|size_t|const char\*)\s+(sparda_\w+)\s*\(", text, re.M)))


def status_string(status):
    return lib.sparda_status_string(int(status)).decode()


sparda_status_string = status_string


def _check(name, status):
    if status != OK:
        raise SpardaError(name, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def num_windows(n_tokens):
    return 0 if n_tokens < WIN_KERNEL else (n_tokens - WIN_KERNEL) // WIN_STRIDE + 1


@dataclass
class Shape:
    """Decode-step geometry (sparda_shape)."""
    n_groups: int = 2
    heads_per_group: int = 16
    head_dim: int = 128
    topk: int = 32
    max_ctx: int = 32768
    max_batch: int = 1
    block: int = BLOCK
    win_kernel: int = WIN_KERNEL
    win_stride: int = WIN_STRIDE

    def c(self):
        return c_shape(self.n_groups, self.heads_per_group, self.head_dim, self.block,
                       self.win_kernel, self.win_stride, self.topk, self.max_ctx, self.max_batch)

    @property
    def w_cap(self):
        return num_windows(self.max_ctx)

    @property
    def kslots(self):
        return self.topk + 2


@dataclass
class LayerKV:
    """One layer's caches (sparda_layer_kv), as torch tensors.

    k, v: bf16 [max_batch, G, max_ctx, d] on the device, or pinned host tensors (on_host).
    ck: bf16 [max_batch, G, w_cap, d] on the device. hot_k, hot_v: bf16
    [max_batch, G, 3, 64, d] on the device for offloaded layers.
    """
    k: torch.Tensor
    v: torch.Tensor
    ck: torch.Tensor
    hot_k: torch.Tensor = None
    hot_v: torch.Tensor = None
    on_host: bool = False

    def c(self):
        return c_layer_kv(self.k.data_ptr(), self.v.data_ptr(), self.ck.data_ptr(),
                          self.hot_k.data_ptr() if self.hot_k is not None else None,
                          self.hot_v.data_ptr() if self.hot_v is not None else None,
                          1 if self.on_host else 0, 0)

    @staticmethod
    def empty(shape, device="cuda", on_host=False):
        G, d = shape.n_groups, shape.head_dim
        kv = (shape.max_batch, G, shape.max_ctx, d)
        if on_host:
            k = torch.empty(kv, dtype=torch.bfloat16, pin_memory=True)
            v = torch.empty(kv, dtype=torch.bfloat16, pin_memory=True)
            hot = (shape.max_batch, G, 3, shape.block, d)
            hk = torch.zeros(hot, dtype=torch.bfloat16, device=device)
            hv = torch.zeros(hot, dtype=torch.bfloat16, device=device)
        else:
            k = torch.empty(kv, dtype=torch.bfloat16, device=device)
            v = torch.empty(kv, dtype=torch.bfloat16, device=device)
            hk = hv = None
        ck = torch.zeros((shape.max_batch, G, shape.w_cap, d), dtype=torch.bfloat16, device=device)
        return LayerKV(k, v, ck, hk, hv, on_host)


def hot_slot(j):
    """Hot-ring slot of block j of an offloaded layer (include/sparda.h, sparda_layer_kv)."""
    return 0 if j == 0 else 1 + (j & 1)


def fill_hot_from_host(layer, n_cached):
    """Set-up after a prefill of an offloaded layer: copy block 0 and the two newest blocks of
    every sequence from the host cache into the hot ring. n_cached[b] = tokens cached so far.
    Plain device copies; not part of the decode step."""
    for b, n in enumerate(n_cached):
        if n < 1:
            continue
        tb = (n - 1) // BLOCK
        for j in sorted({0, tb, max(tb - 1, 0)}):
            rows = slice(j * BLOCK, (j + 1) * BLOCK)
            layer.hot_k[b, :, hot_slot(j)].copy_(layer.k[b, :, rows], non_blocking=False)
            layer.hot_v[b, :, hot_slot(j)].copy_(layer.v[b, :, rows], non_blocking=False)


def workspace(shape, batch, kind, device="cuda"):
    """A zero-filled workspace of the size sparda_workspace_bytes gives."""
    n = sparda_workspace_bytes(shape, batch, kind)
    if n == 0:
        raise SpardaError("sparda_workspace_bytes", ERR_UNSUPPORTED_SHAPE)
    return torch.zeros(n, dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ entry points
def sparda_abi_version():
    return lib.sparda_abi_version()


def sparda_check_shape(shape):
    return lib.sparda_check_shape(ctypes.byref(shape.c()))


def sparda_workspace_bytes(shape, batch, kind):
    return lib.sparda_workspace_bytes(ctypes.byref(shape.c()), int(batch), int(kind))


def sparda_block_scores_offset(shape):
    return lib.sparda_block_scores_offset(ctypes.byref(shape.c()))


def sparda_device_error(clear=True):
    flags = ctypes.c_int32(0)
    _check("sparda_device_error", lib.sparda_device_error(ctypes.byref(flags), 1 if clear else 0))
    return flags.value


def sparda_get_device_status(dev_flag, clear=True, stream=None):
    """Enqueue a stream-ordered copy of the device error word into dev_flag (an int32 tensor
    of one element on the device, or pinned on the host), resetting the word if clear."""
    _check("sparda_get_device_status", lib.sparda_get_device_status(_ptr(dev_flag), 1 if clear else 0,
                                                                      _stream(stream)))


def sparda_prefetch_default_ctas(batch):
    return lib.sparda_prefetch_default_ctas(int(batch))


def sparda_append_kv(shape, layer, k_new, v_new, seq_len, batch, stream=None):
    _check("sparda_append_kv", lib.sparda_append_kv(
        ctypes.byref(shape.c()), ctypes.byref(layer.c()), _ptr(k_new), _ptr(v_new),
        _ptr(seq_len), int(batch), _stream(stream)))


def sparda_compress_keys(shape, layer, seq_len, batch, stream=None):
    _check("sparda_compress_keys", lib.sparda_compress_keys(
        ctypes.byref(shape.c()), ctypes.byref(layer.c()), _ptr(seq_len), int(batch),
        _stream(stream)))


def sparda_forecast_project(W, h, f, stream=None):
    rows, hidden = W.shape
    _check("sparda_forecast_project", lib.sparda_forecast_project(
        _ptr(W), _ptr(h), int(rows), int(hidden), int(h.shape[0]), _ptr(f), _stream(stream)))


def sparda_forecast_select(shape, ck, forecast, seq_len, batch, idx, cnt, ws, stream=None):
    _check("sparda_forecast_select", lib.sparda_forecast_select(
        ctypes.byref(shape.c()), _ptr(ck), _ptr(forecast), _ptr(seq_len), int(batch), _ptr(idx),
        _ptr(cnt), _ptr(ws), ws.numel(), _stream(stream)))


def sparda_sparse_decode_attn(shape, layer, q, idx, cnt, seq_len, batch, out, ws,
                              staging_k=None, staging_v=None, stream=None):
    _check("sparda_sparse_decode_attn", lib.sparda_sparse_decode_attn(
        ctypes.byref(shape.c()), ctypes.byref(layer.c()), _ptr(staging_k), _ptr(staging_v),
        _ptr(q), _ptr(idx), _ptr(cnt), _ptr(seq_len), int(batch), _ptr(out), _ptr(ws),
        ws.numel(), _stream(stream)))


def sparda_attend_and_select(shape, layer, q, idx, cnt, out, ws_attn, ck_next, forecast_next, idx_next,
                             cnt_next, ws_sel, seq_len, batch, staging_k=None, staging_v=None, stream=None):
    _check("sparda_attend_and_select", lib.sparda_attend_and_select(
        ctypes.byref(shape.c()), ctypes.byref(layer.c()), _ptr(staging_k), _ptr(staging_v), _ptr(q), _ptr(idx),
        _ptr(cnt), _ptr(out), _ptr(ws_attn), ws_attn.numel(), _ptr(ck_next), _ptr(forecast_next), _ptr(idx_next),
        _ptr(cnt_next), _ptr(ws_sel), ws_sel.numel(), _ptr(seq_len), int(batch), _stream(stream)))


def sparda_attend_and_score(shape, layer, q, idx, cnt, out, ws_attn, ck_next, forecast_next, ws_scores,
                            seq_len, batch, staging_k=None, staging_v=None, l2_next=None, stream=None):
    """l2_next: an optional tensor the next launches read (pulled into L2 at the end)."""
    _check("sparda_attend_and_score", lib.sparda_attend_and_score(
        ctypes.byref(shape.c()), ctypes.byref(layer.c()), _ptr(staging_k), _ptr(staging_v), _ptr(q), _ptr(idx),
        _ptr(cnt), _ptr(out), _ptr(ws_attn), ws_attn.numel(), _ptr(ck_next), _ptr(forecast_next), _ptr(ws_scores),
        ws_scores.numel(), _ptr(l2_next), l2_next.numel() * l2_next.element_size() if l2_next is not None else 0,
        _ptr(seq_len), int(batch), _stream(stream)))


def sparda_decode_prologue(shape, layer, k_new, v_new, seq_len, batch, ws_scores=None, idx=None, cnt=None,
                           W_next=None, h=None, forecast_next=None, stream=None):
    """Layer L's top-k (from ws_scores, if given), append, and forecast for layer L+1 (if
    W_next is given) in one launch."""
    hidden = int(W_next.shape[1]) if W_next is not None else 0
    _check("sparda_decode_prologue", lib.sparda_decode_prologue(
        ctypes.byref(shape.c()), ctypes.byref(layer.c()), _ptr(k_new), _ptr(v_new), _ptr(ws_scores),
        ws_scores.numel() if ws_scores is not None else 0, _ptr(idx), _ptr(cnt), _ptr(W_next), _ptr(h), hidden,
        _ptr(forecast_next), _ptr(seq_len), int(batch), _stream(stream)))


def sparda_prefetch_blocks(shape, layer, idx, cnt, seq_len, batch, staging_k, staging_v,
                           n_ctas=0, stream=None):
    _check("sparda_prefetch_blocks", lib.sparda_prefetch_blocks(
        ctypes.byref(shape.c()), ctypes.byref(layer.c()), _ptr(idx), _ptr(cnt), _ptr(seq_len),
        int(batch), _ptr(staging_k), _ptr(staging_v), int(n_ctas), _stream(stream)))


def sparda_forecast_score(shape, ck, forecast, seq_len, batch, ws, stream=None):
    """Block scores of the Forecast selector without the top-k, into the select workspace ws
    (for sparda_decode_prologue's ws_scores)."""
    _check("sparda_forecast_score", lib.sparda_forecast_score(
        ctypes.byref(shape.c()), _ptr(ck), _ptr(forecast), _ptr(seq_len), int(batch), _ptr(ws), ws.numel(),
        _stream(stream)))


def sparda_copy(dst, src, stream=None):
    """Device-side copy of src into dst (same byte size, each contiguous): device tensors or
    pinned host tensors (see include/sparda.h)."""
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes or not dst.is_contiguous() or not src.is_contiguous():
        raise ValueError("sparda_copy needs two contiguous tensors of the same byte size")
    _check("sparda_copy", lib.sparda_copy(_ptr(dst), _ptr(src), nbytes, _stream(stream)))


def sparda_multihead_select(shape, ck, q, seq_len, batch, idx, cnt, ws, stream=None):
    _check("sparda_multihead_select", lib.sparda_multihead_select(
        ctypes.byref(shape.c()), _ptr(ck), _ptr(q), _ptr(seq_len), int(batch), _ptr(idx),
        _ptr(cnt), _ptr(ws), ws.numel(), _stream(stream)))


def sparda_forecast_select_static(shape, ck, forecast, seq_len, batch, idx, cnt, stream=None):
    """sparda_forecast_select without a workspace: for callers that may not allocate device
    memory. Its scratch is a fixed array inside the library (see include/sparda.h)."""
    _check("sparda_forecast_select_static", lib.sparda_forecast_select_static(
        ctypes.byref(shape.c()), _ptr(ck), _ptr(forecast), _ptr(seq_len), int(batch), _ptr(idx),
        _ptr(cnt), _stream(stream)))


# ------------------------------------------------------------------ chunked prefill
def sparda_prefill_forecast_select(shape, ck, forecast, seq_len, batch, idx, cnt, ws, stream=None):
    """Per-chunk selections of a prompt by the Forecast selector. forecast: bf16
    [max_batch, max_ctx, G, d]; idx: int32 [B, G, max_ctx/64, topk+2]; cnt: int32
    [B, G, max_ctx/64]; ws: a WS_PREFILL workspace."""
    _check("sparda_prefill_forecast_select", lib.sparda_prefill_forecast_select(
        ctypes.byref(shape.c()), _ptr(ck), _ptr(forecast), _ptr(seq_len), int(batch), _ptr(idx), _ptr(cnt),
        _ptr(ws), ws.numel(), _stream(stream)))


def sparda_prefill_multihead_select(shape, ck, q, seq_len, batch, idx, cnt, ws, stream=None):
    """Per-chunk selections of a prompt by the baseline multi-head selector. q: bf16
    [max_batch, max_ctx, G*H, d]; outputs as sparda_prefill_forecast_select."""
    _check("sparda_prefill_multihead_select", lib.sparda_prefill_multihead_select(
        ctypes.byref(shape.c()), _ptr(ck), _ptr(q), _ptr(seq_len), int(batch), _ptr(idx), _ptr(cnt),
        _ptr(ws), ws.numel(), _stream(stream)))


def sparda_prefill_attn(shape, layer, q, idx, cnt, seq_len, batch, out, stream=None):
    """Causal block-sparse prefill attention of a resident layer over the per-chunk
    selections. q, out: bf16 [max_batch, max_ctx, G*H, d]."""
    _check("sparda_prefill_attn", lib.sparda_prefill_attn(
        ctypes.byref(shape.c()), ctypes.byref(layer.c()), _ptr(q), _ptr(idx), _ptr(cnt), _ptr(seq_len),
        int(batch), _ptr(out), _stream(stream)))


# ------------------------------------------------------------------ cross-step block cache
class BlockCache:
    """The block cache of one offloaded layer (include/sparda.h): n_cache HBM slots per
    (sequence, group) holding blocks gathered at earlier steps, the block each slot holds
    (-1: none), the slot of each idx entry, and the gather's scratch."""

    def __init__(self, shape, n_cache=None, device="cuda"):
        n = shape.kslots if n_cache is None else int(n_cache)
        B, G = shape.max_batch, shape.n_groups
        self.n_cache = n
        self.k = torch.zeros((B, G, n, shape.block, shape.head_dim), dtype=torch.bfloat16, device=device)
        self.v = torch.zeros_like(self.k)
        self.blocks = torch.full((B, G, n), -1, dtype=torch.int32, device=device)
        self.slot = torch.full((B, G, shape.kslots), -1, dtype=torch.int32, device=device)
        self.fetch = torch.full((B, G, n), -1, dtype=torch.int32, device=device)

    def reset(self):
        self.blocks.fill_(-1)


def sparda_prefetch_blocks_cached(shape, layer, idx, cnt, seq_len, batch, cache, stats=None, n_ctas=0,
                                  stream=None):
    """Gather of the selected blocks not yet in `cache` (a BlockCache); stats: optional int64
    tensor [2] on the device accumulating hits and misses."""
    _check("sparda_prefetch_blocks_cached", lib.sparda_prefetch_blocks_cached(
        ctypes.byref(shape.c()), ctypes.byref(layer.c()), _ptr(idx), _ptr(cnt), _ptr(seq_len), int(batch),
        _ptr(cache.k), _ptr(cache.v), _ptr(cache.blocks), int(cache.n_cache), _ptr(cache.slot), _ptr(cache.fetch),
        _ptr(stats), int(n_ctas), _stream(stream)))


def sparda_sparse_decode_attn_cached(shape, layer, cache, q, idx, cnt, seq_len, batch, out, ws, stream=None):
    """Attention of an offloaded layer over its selected blocks, read from `cache`."""
    _check("sparda_sparse_decode_attn_cached", lib.sparda_sparse_decode_attn_cached(
        ctypes.byref(shape.c()), ctypes.byref(layer.c()), _ptr(cache.k), _ptr(cache.v), int(cache.n_cache),
        _ptr(cache.slot), _ptr(q), _ptr(idx), _ptr(cnt), _ptr(seq_len), int(batch), _ptr(out), _ptr(ws),
        ws.numel(), _stream(stream)))


def sparda_prefetch_blocks_copy_engine(shape, layer, idx_host, cnt_host, seq_len_host, batch, staging_k, staging_v,
                                       stream=None):
    """The gather by one cudaMemcpyAsync per run of consecutive selected blocks; the selection
    (idx_host, cnt_host, seq_len_host) must be int32 CPU tensors. Returns the number of copies
    issued."""
    for t in (idx_host, cnt_host, seq_len_host):
        if t.device.type != "cpu" or t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError("the copy-engine gather takes the selection as contiguous int32 CPU tensors")
    n = ctypes.c_int32(0)
    _check("sparda_prefetch_blocks_copy_engine", lib.sparda_prefetch_blocks_copy_engine(
        ctypes.byref(shape.c()), ctypes.byref(layer.c()), ctypes.c_void_p(idx_host.data_ptr()),
        ctypes.c_void_p(cnt_host.data_ptr()), ctypes.c_void_p(seq_len_host.data_ptr()), int(batch),
        _ptr(staging_k), _ptr(staging_v), ctypes.byref(n), _stream(stream)))
    return n.value
