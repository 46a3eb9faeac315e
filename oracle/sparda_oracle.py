"""Plain, slow fp64 CPU oracle of the SparDA forecast-driven block-sparse decode step and of
its chunked prefill.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this module. The product path (the CUDA library under
``block_sparse_attention_forecast_gb300/`` and its Python binding) never imports, calls or
links it, and this module imports nothing from the product. It shares no code, table or
helper with the GPU path.

Sources. The method is described only in prose by three web pages about the paper
"SparDA: Sparse Decoupled Attention for Efficient Long-Context LLM Inference":

  [thread]     bittide.aicompass.dev article 75eb008a (a thread on SparDA, followed by the
               translated arXiv abstract);
  [techwalker] techwalker.com "NVIDIA与MIT联手：让超长文本AI助手的'记忆搜索'快了5倍多",
               sections 一 (the problem), 二 (the Forecast idea), 三 (implementation),
               四 (training), 五 (experiments);
  [10100]      10100.com article 150198800 "不是我硬件不好 是你软件架构有硬伤",
               sections "先把痛点讲透" and "SparDA 的解法".

The pages print no equations, code, block size or top-k. Every step below states the
passage it follows and, where the pages are silent, the reading taken:

  * compressed keys: the mean of each key window of kernel 32 / stride 16 ([techwalker] §四
    names this inference-time key compression window; "mean" is the reading taken), stored
    as bfloat16 like the keys themselves;
  * forecast scoring: ONE forecast vector per GQA group scores each compressed key by a plain
    dot product, with no softmax and no per-query-head loop ([thread], the paragraph on one
    Forecast head per GQA group; [techwalker] §二, first benefit; [10100] "SparDA 的解法");
  * window scores are max-pooled onto 64-token KV blocks, taking every window that overlaps
    the block (max-pooling from a finer to a coarser grid is the operation [techwalker] §四
    describes for its training targets; block 64 is this library's constant);
  * block selection keeps the top-k scored blocks plus two always-kept blocks, block 0 and
    the block holding the current token ([thread] "score the KV cache by block, keep the top-k
    blocks"; the forced blocks are a reading);
  * block-sparse attention: the decode query of every head of the group attends only the
    tokens of the selected blocks, with ordinary scaled softmax attention ([thread], "layer
    L+1's own queries attend the selected blocks"; [techwalker] §六: SparDA leaves the sparse
    attention computation itself unchanged);
  * the baseline (query-driven) selector: every query head of the group scores every
    candidate, a softmax per head, then a sum over the group ([thread], the paragraph on the
    standard selector; [10100] "先把痛点讲透");
  * the forecast projection: a fourth per-layer linear projection of the hidden state, one
    128-wide head per KV group ([thread] "each layer now outputs four projections";
    [techwalker] §二 and §四 (33.5M parameters, 0.41%));
  * lookahead: layer L's forecast selects layer L+1's blocks; layer 0 has no earlier
    forecast and selects its own blocks from a same-layer forecast ([thread]; [techwalker]
    §三, last paragraph).

Everything is computed in float64 from the exact bfloat16 input values. bfloat16 rounding
(round to nearest, ties to even) is written out below from the format's definition.
"""
from __future__ import annotations

import math

import numpy as np

# Sizes the decode step works with (the pages fix the window; block 64 is a chosen constant).
BLOCK = 64          # tokens per KV block
WIN_KERNEL = 32     # tokens per compression window ([techwalker] §四: kernel 32)
WIN_STRIDE = 16     # window stride ([techwalker] §四: stride 16)


# --------------------------------------------------------------------------------------
# bfloat16 rounding, from the format's definition
# --------------------------------------------------------------------------------------
def bf16_round(x):
    """Round float64 values to the nearest bfloat16 value, ties to even; returns float64.

    bfloat16 keeps float32's 8 exponent bits and 7 stored fraction bits: 8 significant bits
    for normal numbers (|x| >= 2^-126) and a fixed spacing of 2^-133 below that. The spacing
    of representable values in [2^e, 2^(e+1)) is therefore 2^(max(e, -126) - 7); rounding to
    that grid with ties to even is np.rint (IEEE round-half-even) of x / spacing. Results of
    magnitude 2^128 or more overflow to infinity.
    """
    x = np.asarray(x, dtype=np.float64)
    finite = np.isfinite(x)
    ax = np.where(finite, np.abs(x), 1.0)
    _, E = np.frexp(ax)                       # ax = m * 2^E, m in [0.5, 1)
    e = np.maximum(E - 1, -126)               # 2^e <= ax < 2^(e+1), clamped to the normal floor
    spacing = np.ldexp(1.0, e - 7)
    r = np.rint(np.where(finite, x, 0.0) / spacing) * spacing
    r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, x), r)
    return np.where(finite, r, x)


# --------------------------------------------------------------------------------------
# Compressed keys
# --------------------------------------------------------------------------------------
def num_windows(n_tokens, kernel=WIN_KERNEL, stride=WIN_STRIDE):
    """Number of complete compression windows over the first ``n_tokens`` tokens.

    Window i covers tokens [stride*i, stride*i + kernel). Only complete windows exist (a
    reading: the pages say nothing about partial windows), so one new window appears every
    ``stride`` tokens once ``kernel`` tokens are cached.
    """
    if n_tokens < kernel:
        return 0
    return (n_tokens - kernel) // stride + 1


def compress_keys(K, n_windows, kernel=WIN_KERNEL, stride=WIN_STRIDE):
    """Compressed keys of one (sequence, KV group): ck[i] = bf16(mean of keys in window i).

    K: [T, d] float64 holding bfloat16 values. Window i averages keys stride*i ..
    stride*i + kernel - 1 ([techwalker] §四: the inference-time key compression window has
    kernel 32 and stride 16). The mean is exact in float64 for bfloat16 inputs of ordinary
    range and is then rounded to bfloat16, the storage type of the keys.
    """
    K = np.asarray(K, dtype=np.float64)
    d = K.shape[1]
    ck = np.empty((n_windows, d), dtype=np.float64)
    for i in range(n_windows):
        window = K[stride * i: stride * i + kernel]
        assert window.shape[0] == kernel, "window runs past the cached tokens"
        ck[i] = bf16_round(window.sum(axis=0) / kernel)
    return ck


# --------------------------------------------------------------------------------------
# Forecast selector
# --------------------------------------------------------------------------------------
def forecast_scores(ck, f):
    """Window scores of the Forecast selector: s[i] = <f, ck[i]>, no softmax, no scale.

    One forecast vector f per GQA group scores every compressed key directly ([thread]: one
    Forecast head per GQA group, skipping the softmax; [techwalker] §二).
    """
    return np.asarray(ck, dtype=np.float64) @ np.asarray(f, dtype=np.float64)


def multihead_scores(q_group, ck, scale=None):
    """Window scores of the baseline query-driven selector.

    Every query head h of the group scores every compressed key, each head's scores go
    through a softmax over the windows, and the per-head probabilities are summed over the
    group ([thread], the paragraph on the standard selector; [10100] "先把痛点讲透"). The
    scores use the attention scale 1/sqrt(d) (a reading: the usual attention logit scale).
    """
    q_group = np.asarray(q_group, dtype=np.float64)
    ck = np.asarray(ck, dtype=np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(q_group.shape[1])
    z = (q_group @ ck.T) * scale                      # [H, W]
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p = p / p.sum(axis=1, keepdims=True)              # softmax over windows, per head
    return p.sum(axis=0)                              # sum over the heads of the group


def window_block_overlap(i, j, block=BLOCK, kernel=WIN_KERNEL, stride=WIN_STRIDE):
    """True when window i (tokens [stride*i, stride*i+kernel)) overlaps block j."""
    w0, w1 = stride * i, stride * i + kernel
    b0, b1 = block * j, block * (j + 1)
    return w0 < b1 and w1 > b0


def pool_to_blocks(s, n_blocks, block=BLOCK, kernel=WIN_KERNEL, stride=WIN_STRIDE,
                   mode="overlap"):
    """Block scores: S[j] = max of the window scores over the windows that overlap block j.

    ``mode="overlap"`` (the reading used throughout) takes every window that shares a token
    with the block; ``mode="inside"`` takes only windows lying wholly in the block (the
    alternative reading, kept for comparison). A block with no scored window gets -inf.
    For speed the loop over windows of block j only visits i in
    [(block*j - kernel) // stride, block*(j+1) // stride], a range that contains every
    window touching the block; each visited window is still tested by the predicate.
    """
    s = np.asarray(s, dtype=np.float64)
    S = np.full(n_blocks, -np.inf)
    for j in range(n_blocks):
        lo = max(0, (block * j - kernel) // stride)
        hi = min(s.shape[0], (block * (j + 1)) // stride + 1)
        for i in range(lo, hi):
            if mode == "overlap":
                take = window_block_overlap(i, j, block, kernel, stride)
            elif mode == "inside":
                take = stride * i >= block * j and stride * i + kernel <= block * (j + 1)
            else:
                raise ValueError(mode)
            if take and s[i] > S[j]:
                S[j] = s[i]
    return S


def tail_block(T, block=BLOCK):
    """Index of the block holding the current (last) token of a T-token context."""
    return (T - 1) // block


def select_blocks(S, T, k, block=BLOCK, forced_in_k=False):
    """Top-k block selection with the always-kept blocks.

    The forced set is {0, tail block}. The remaining blocks of the context are ranked by
    block score, higher first, a tie going to the lower block index, and the first k are
    kept (or the first k - |forced| when ``forced_in_k``, the alternative reading). Returns
    the selected block indices sorted ascending.
    """
    S = np.asarray(S, dtype=np.float64)
    tb = tail_block(T, block)
    forced = sorted({0, tb})
    cand = np.array([j for j in range(tb + 1) if j not in forced], dtype=np.int64)
    n_take = k - len(forced) if forced_in_k else k
    n_take = max(0, min(n_take, cand.size))
    if cand.size:
        order = np.lexsort((cand, -S[cand]))          # primary: score desc; then index asc
        chosen = cand[order[:n_take]]
    else:
        chosen = cand
    return sorted(set(forced) | set(int(j) for j in chosen))


def topk_boundary(S, T, k, block=BLOCK):
    """The k-th and (k+1)-th largest candidate block scores (None where absent).

    Used to decide whether a selection is unique: when the two are close the k-th slot has
    several correct answers.
    """
    tb = tail_block(T, block)
    forced = {0, tb}
    vals = np.sort(np.array([S[j] for j in range(tb + 1) if j not in forced]))[::-1]
    kth = vals[k - 1] if 0 < k <= vals.size else None
    k1th = vals[k] if k < vals.size else None
    return kth, k1th


# --------------------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------------------
def selected_tokens(sel, T, block=BLOCK):
    """Token positions of the selected blocks that lie inside the T-token context."""
    toks = []
    for j in sel:
        toks.extend(range(block * j, min(block * (j + 1), T)))
    return np.array(toks, dtype=np.int64)


def block_sparse_attention(q_group, K, V, sel, T, block=BLOCK, scale=None):
    """Decode attention of all query heads of a group over the selected blocks only.

    q_group: [H, d]; K, V: [>=T, d]. For every head, o = sum_t softmax_t(q.k_t * scale) v_t
    over the tokens t < T of the selected blocks ([thread]: the next layer's own query runs
    sparse attention over the chosen blocks). Scale 1/sqrt(d).
    """
    q_group = np.asarray(q_group, dtype=np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(q_group.shape[1])
    toks = selected_tokens(sel, T, block)
    Kt = np.asarray(K, dtype=np.float64)[toks]
    Vt = np.asarray(V, dtype=np.float64)[toks]
    z = (q_group @ Kt.T) * scale                      # [H, n]
    z = z - z.max(axis=1, keepdims=True)
    w = np.exp(z)
    return (w @ Vt) / w.sum(axis=1, keepdims=True)


def dense_causal_attention(q_group, K, V, T, scale=None):
    """Dense decode attention over every cached token t < T (written independently of the
    block-sparse routine, as a log-sum-exp per head, to pin it)."""
    q_group = np.asarray(q_group, dtype=np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(q_group.shape[1])
    K = np.asarray(K, dtype=np.float64)[:T]
    V = np.asarray(V, dtype=np.float64)[:T]
    out = np.empty((q_group.shape[0], V.shape[1]))
    for h in range(q_group.shape[0]):
        logits = K @ q_group[h] * scale
        lse = np.logaddexp.reduce(logits)
        out[h] = np.exp(logits - lse) @ V
    return out


# --------------------------------------------------------------------------------------
# Forecast projection
# --------------------------------------------------------------------------------------
def forecast_project(W, h):
    """Forecast vectors from a hidden state: bf16(W @ h).

    W: [G*d, hidden] (row g*d + c is component c of group g's forecast head), h: [hidden].
    The fourth per-layer projection ([thread]; [techwalker] §二), computed exactly in
    float64 and rounded to bfloat16, the storage type of the projection outputs.
    """
    return bf16_round(np.asarray(W, dtype=np.float64) @ np.asarray(h, dtype=np.float64))


# --------------------------------------------------------------------------------------
# One (sequence, group) selection and one whole decode step
# --------------------------------------------------------------------------------------
def forecast_select_one(K, f, T, k, block=BLOCK, kernel=WIN_KERNEL, stride=WIN_STRIDE,
                        mode="overlap", forced_in_k=False, return_scores=False):
    """Select the blocks of one (sequence, group) for a T-token context.

    The selector scores the compressed keys of the tokens cached before the current one
    (windows complete within the first T-1 tokens): under lookahead the target layer's key
    for the current token does not exist yet when the previous layer's forecast selects its
    blocks ([thread]: the block set is known while the current layer still computes). The
    current token lies in the tail block, which is always kept.
    """
    W = num_windows(T - 1, kernel, stride)
    ck = compress_keys(K, W, kernel, stride)
    s = forecast_scores(ck, f)
    nb = tail_block(T, block) + 1
    S = pool_to_blocks(s, nb, block, kernel, stride, mode)
    sel = select_blocks(S, T, k, block, forced_in_k)
    if return_scores:
        return sel, S
    return sel


def decode_step(layers, W_self0, W_next, h, q, k_new, v_new, p, topk, heads_per_group,
                block=BLOCK, kernel=WIN_KERNEL, stride=WIN_STRIDE):
    """One decode step of the forecast-driven block-sparse stack at token position p.

    layers[L] = (K, V): float64 [B, G, >=p+1, d] caches holding tokens 0..p-1.
    W_self0: [G*d, hidden], layer 0's same-layer forecast head; W_next[L] (L < n_layers-1):
    [G*d, hidden], layer L's forecast head for layer L+1. h[L]: [B, hidden]; q[L]:
    [B, G*H, d]; k_new[L], v_new[L]: [B, G, d].

    Per layer L (the order of [thread] and [techwalker] §二-§三): store the token's key and
    value at position p; layer 0 selects its own blocks from its same-layer forecast;
    layer L's forecast selects layer L+1's blocks; layer L attends its selected blocks with
    its own queries. Returns (sel, out): sel[L][b][g] is the sorted block list that layer L
    attended, out[L] is [B, G*H, d].
    """
    n_layers = len(layers)
    T = p + 1
    B, G = layers[0][0].shape[:2]
    Hh = heads_per_group
    sel = [None] * n_layers
    out = [None] * n_layers
    for L in range(n_layers):
        K, V = layers[L]
        K[:, :, p] = k_new[L]
        V[:, :, p] = v_new[L]
        d = K.shape[3]
        if L == 0:
            f0 = np.stack([forecast_project(W_self0, h[0][b]).reshape(G, d) for b in range(B)])
            sel[0] = [[forecast_select_one(K[b, g], f0[b, g], T, topk, block, kernel, stride)
                       for g in range(G)] for b in range(B)]
        if L + 1 < n_layers:
            Kn = layers[L + 1][0]
            f = np.stack([forecast_project(W_next[L], h[L][b]).reshape(G, d) for b in range(B)])
            sel[L + 1] = [[forecast_select_one(Kn[b, g], f[b, g], T, topk, block, kernel,
                                               stride) for g in range(G)] for b in range(B)]
        o = np.empty(q[L].shape)
        for b in range(B):
            for g in range(G):
                qg = q[L][b, g * Hh:(g + 1) * Hh]
                o[b, g * Hh:(g + 1) * Hh] = block_sparse_attention(qg, K[b, g], V[b, g],
                                                                   sel[L][b][g], T, block)
        out[L] = o
    return sel, out


# --------------------------------------------------------------------------------------
# Prefill: chunked queries
# --------------------------------------------------------------------------------------
# The pages measure prefill as well as decode ([thread] and the abstract: up to 1.25x faster
# prefill; [techwalker] §五, the per-layer breakdown: in prefill the block-sparse attention
# dominates, the block selection grows with the context and is close to it at 128K, and the
# Forecast indexer cuts the selection cost by up to 2.5x while the attention is unchanged;
# [10100]: in prefill all keys are already on the GPU, so the gain is the cheaper selection
# alone). They do not spell the prefill selection out. The readings taken here:
#
#   * the prompt is processed in chunks of 64 query tokens (one KV block); chunk c holds the
#     tokens [64c, 64c + 64) of the prompt, the last chunk possibly fewer;
#   * the tokens of a chunk share one block selection, so that the block-sparse attention
#     of the chunk reads each selected block once;
#   * the selection of chunk c scores the compressed keys complete before the chunk starts
#     (the windows within its first 64c tokens), as a decode step scores the windows complete
#     before its current token; block 0 and the chunk's own block c are always kept, and the
#     top-k of the blocks 1 .. c-1 is added;
#   * the Forecast selector scores a window by the sum over the chunk's tokens of the decode
#     score (each token's forecast vector dotted with the compressed key, no softmax, no
#     scale); the baseline selector sums over the chunk's tokens what it sums over the
#     group's heads in decode (each (token, head) query's softmax over the windows);
#   * every query token attends the tokens of its chunk's selected blocks up to and including
#     its own position (causal within the chunk's own block).
def prefill_num_chunks(T, block=BLOCK):
    """Chunks of a T-token prompt."""
    return (T + block - 1) // block


def prefill_chunk_windows(c, block=BLOCK, kernel=WIN_KERNEL, stride=WIN_STRIDE):
    """Windows complete before chunk c starts: those within its first block*c tokens."""
    return num_windows(block * c, kernel, stride)


def prefill_forecast_scores(F_chunk, ck, c, block=BLOCK):
    """Window scores of chunk c under the Forecast selector.

    F_chunk: [n_tok, d], the forecast vectors of the chunk's tokens (one head of the group);
    ck: the group's compressed keys. s[i] = sum over the chunk's tokens t of <f_t, ck[i]>,
    for the windows i complete before the chunk.
    """
    W = prefill_chunk_windows(c, block)
    per_token = np.asarray(F_chunk, dtype=np.float64) @ np.asarray(ck, dtype=np.float64)[:W].T   # [n_tok, W]
    return per_token.sum(axis=0)


def prefill_multihead_scores(Q_chunk, ck, c, scale=None, block=BLOCK):
    """Window scores of chunk c under the baseline selector.

    Q_chunk: [n_tok, H, d], the query heads of the group for each token of the chunk. Every
    (token, head) query gets its own softmax over the windows complete before the chunk (its
    logits scaled by 1/sqrt(d)), and the probabilities are summed over the chunk's tokens and
    the group's heads.
    """
    Q_chunk = np.asarray(Q_chunk, dtype=np.float64)
    W = prefill_chunk_windows(c, block)
    if W == 0:
        return np.zeros(0)
    n_tok, H, d = Q_chunk.shape
    total = np.zeros(W)
    for t in range(n_tok):
        total += multihead_scores(Q_chunk[t], np.asarray(ck)[:W], scale)
    return total


def prefill_select(S, c, k, block=BLOCK):
    """Blocks of chunk c: {0, c} and the top-k of the blocks 1 .. c-1 by S (ties to the lower
    block), ascending. The rule is the decode step's, for a context whose current token lies
    in block c."""
    return select_blocks(S, block * c + 1, k, block)


def prefill_select_all(ck, per_chunk_queries, T, k, selector="forecast", block=BLOCK):
    """Selections of every chunk of a T-token prompt for one (sequence, group).

    per_chunk_queries(c) returns the chunk's forecast vectors [n_tok, d] ("forecast") or its
    queries [n_tok, H, d] ("multihead"). Returns (sel, S): the block lists and the block
    scores of each chunk.
    """
    sel, S = [], []
    for c in range(prefill_num_chunks(T, block)):
        if selector == "forecast":
            s = prefill_forecast_scores(per_chunk_queries(c), ck, c, block)
        else:
            s = prefill_multihead_scores(per_chunk_queries(c), ck, c, block=block)
        Sc = pool_to_blocks(s, c + 1, block)
        S.append(Sc)
        sel.append(prefill_select(Sc, c, k, block))
    return sel, S


def prefill_block_sparse_attention(Q, K, V, sel, T, block=BLOCK, scale=None):
    """Causal block-sparse prefill attention of one (sequence, group).

    Q: [T, H, d], the group's query heads for every prompt token; K, V: [>=T, d]; sel[c]: the
    blocks of chunk c. Token t of chunk c = t // block attends, for every head, the tokens
    t' <= t of its chunk's blocks. Returns [T, H, d].
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(Q.shape[2])
    out = np.empty(Q.shape)
    for t in range(T):
        toks = selected_tokens(sel[t // block], t + 1, block)          # tokens <= t
        z = (Q[t] @ K[toks].T) * scale                                 # [H, n]
        z = z - z.max(axis=1, keepdims=True)
        w = np.exp(z)
        out[t] = (w @ V[toks]) / w.sum(axis=1, keepdims=True)
    return out


def dense_causal_prefill_attention(Q, K, V, T, scale=None):
    """Dense causal prefill attention: token t attends every token t' <= t (written
    separately from the block-sparse routine, per head as a log-sum-exp, to pin it)."""
    Q = np.asarray(Q, dtype=np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(Q.shape[2])
    out = np.empty(Q.shape)
    for t in range(T):
        out[t] = dense_causal_attention(Q[t], K, V, t + 1, scale)
    return out
