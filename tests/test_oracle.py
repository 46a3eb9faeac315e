"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test checks one part of the oracle against a closed form, a hand-derived value, a
library routine in a case where it computes the same thing, an invariant of the method, or
a brute-force enumeration, chosen so that a plausible slip (a wrong window offset or
divisor, a transposed operand, a missing scale, a dropped softmax, a wrong pooling range, an
inverted tie-break, a forced block counted inside k, a lookahead wired to the wrong layer)
fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import sparda_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- bfloat16 rounding
def test_bf16_round_matches_torch_on_float32_values():
    # torch's float32 -> bfloat16 conversion rounds to nearest even; on float32 inputs the
    # float64 rounding must agree with it bit for bit.
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-30).astype(np.float32),
        (rng.standard_normal(20000) * 1e30).astype(np.float32),
        rng.integers(-70000, 70000, 20000).astype(np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_round(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_round_ties_and_edges():
    e = 2.0 ** -8
    assert O.bf16_round(1 + e) == 1.0                       # tie, even neighbour is 1
    assert O.bf16_round(1 + 3 * e) == 1 + 4 * e              # tie, even neighbour is up
    assert O.bf16_round(1 + e + 2.0 ** -30) == 1 + 2 * e     # just above the tie
    assert O.bf16_round(-(1 + 3 * e)) == -(1 + 4 * e)
    assert O.bf16_round(3 * 2.0 ** -134) == 2.0 ** -132       # subnormal tie -> even
    assert O.bf16_round(2.0 ** -133) == 2.0 ** -133
    assert np.isinf(O.bf16_round(2.0 ** 128))
    big = (2 - 2.0 ** -7) * 2.0 ** 127                       # largest finite bfloat16
    assert O.bf16_round(big) == big
    assert np.isinf(O.bf16_round(big + 2.0 ** 119))          # halfway to 2^128 -> inf


# ---------------------------------------------------------------- compressed keys
def test_num_windows_hand_values():
    assert [O.num_windows(n) for n in (0, 31, 32, 47, 48, 63, 64)] == [0, 0, 1, 1, 2, 2, 3]
    assert O.num_windows(4095) == 254 and O.num_windows(4096) == 255
    assert O.num_windows(32767) == 2046 and O.num_windows(131072) == 8191


def test_compress_keys_constant_and_ramp():
    K = np.full((96, 3), 1.25)
    assert np.array_equal(O.compress_keys(K, 5), np.full((5, 3), 1.25))
    # K[t] = t: window i averages 16i .. 16i+31, whose mean is 16i + 15.5
    K = np.repeat(np.arange(160, dtype=np.float64)[:, None], 2, axis=1)
    ck = O.compress_keys(K, 9)
    want = O.bf16_round(16 * np.arange(9) + 15.5)
    assert np.array_equal(ck[:, 0], want) and np.array_equal(ck[:, 1], want)
    assert ck[3, 0] == 63.5                                   # exactly representable


def test_compress_keys_window_straddling_two_blocks():
    K = np.concatenate([np.ones((64, 4)), 3 * np.ones((64, 4))])
    ck = O.compress_keys(K, 7)
    assert np.array_equal(ck[:, 0], [1, 1, 1, 2, 3, 3, 3])


# ---------------------------------------------------------------- scoring / pooling
def test_forecast_scores_small_integers():
    ck = np.array([[1, 2, 3], [-1, 0, 4], [0, 0, 0]], dtype=np.float64)
    f = np.array([2, -1, 1], dtype=np.float64)
    assert np.array_equal(O.forecast_scores(ck, f), [3, 2, 0])


def test_overlap_rule_is_windows_4j_minus_1_to_4j_plus_3():
    for j in range(30):
        for i in range(130):
            assert O.window_block_overlap(i, j) == (4 * j - 1 <= i <= 4 * j + 3)


def test_pooling_range_restriction_equals_full_scan():
    rng = np.random.default_rng(1)
    for W, nb in ((1, 2), (11, 4), (254, 64), (255, 64)):
        s = rng.standard_normal(W)
        for mode in ("overlap", "inside"):
            full = np.full(nb, -np.inf)
            for j in range(nb):
                for i in range(W):
                    if mode == "overlap":
                        ok = O.window_block_overlap(i, j)
                    else:
                        ok = 16 * i >= 64 * j and 16 * i + 32 <= 64 * (j + 1)
                    if ok:
                        full[j] = max(full[j], s[i])
            assert np.array_equal(O.pool_to_blocks(s, nb, mode=mode), full)


def test_single_hot_window_marks_exactly_its_blocks():
    for i in range(40):
        s = np.zeros(40)
        s[i] = 1.0
        S = O.pool_to_blocks(s, 12)
        hot = [j for j in range(12) if S[j] == 1.0]
        assert hot == [j for j in range(12) if 4 * j - 1 <= i <= 4 * j + 3]


def test_pooling_is_monotone():
    rng = np.random.default_rng(2)
    for _ in range(50):
        s = rng.standard_normal(61)
        S0 = O.pool_to_blocks(s, 16)
        s2 = s.copy()
        s2[rng.integers(61)] += abs(rng.standard_normal()) + 1e-3
        S1 = O.pool_to_blocks(s2, 16)
        assert np.all(S1 >= S0)


# ---------------------------------------------------------------- top-k selection
def _brute_select(S, T, k):
    """Independent brute force: a candidate is chosen iff fewer than k candidates beat it
    (a higher score, or an equal score at a lower index)."""
    tb = (T - 1) // 64
    forced = {0, tb}
    cand = [j for j in range(tb + 1) if j not in forced]
    chosen = set()
    for j in cand:
        beaten_by = sum(1 for i in cand if S[i] > S[j] or (S[i] == S[j] and i < j))
        if beaten_by < k:
            chosen.add(j)
    return sorted(forced | chosen)


def test_topk_brute_force_equals_sort():
    rng = np.random.default_rng(3)
    for trial in range(300):
        T = int(rng.integers(1, 64 * 40))
        nb = (T - 1) // 64 + 1
        S = rng.integers(-4, 5, nb).astype(np.float64)     # many ties on purpose
        k = int(rng.integers(0, 12))
        assert O.select_blocks(S, T, k) == _brute_select(S, T, k)


def test_topk_forced_blocks_tie_break_and_sizes():
    S = np.array([0.0, 5, 5, 1, 9, 9])                     # T in block 5 -> forced {0, 5}
    T = 5 * 64 + 10
    # candidates 1..4 score 5, 5, 1, 9 (block 5's 9 is forced, not a candidate)
    assert O.select_blocks(S, T, 1) == [0, 4, 5]
    assert O.select_blocks(S, T, 2) == [0, 1, 4, 5]        # tie 5 vs 5 -> lower index 1
    assert O.select_blocks(S, T, 3) == [0, 1, 2, 4, 5]
    assert O.select_blocks(S, T, 10) == [0, 1, 2, 3, 4, 5]  # k >= candidates -> all
    assert O.select_blocks(S, T, 0) == [0, 5]
    assert O.select_blocks(S, 64, 4) == [0]                 # tail is block 0
    assert O.select_blocks(S, 65, 4) == [0, 1]
    # forced blocks counted inside k (the alternative reading) keeps k blocks in total
    assert O.select_blocks(S, T, 3, forced_in_k=True) == [0, 4, 5]


def test_topk_picks_highest_scores_not_lowest():
    S = np.array([0.0, 1, 7, 3, 0])
    assert O.select_blocks(S, 4 * 64 + 1, 1) == [0, 2, 4]


def test_topk_boundary_hand_cases():
    # T in block 5 -> forced {0, 5}; candidates 1..4 score 5, 2, 1, 9. Block 0 (100) and the
    # tail block 5 (50) are the two largest scores, and must not count as candidates.
    S = np.array([100.0, 5, 2, 1, 9, 50])
    T = 5 * 64 + 10
    assert O.topk_boundary(S, T, 1) == (9.0, 5.0)
    assert O.topk_boundary(S, T, 2) == (5.0, 2.0)
    assert O.topk_boundary(S, T, 3) == (2.0, 1.0)
    # k = number of candidates: a k-th but no (k+1)-th; k beyond it: neither
    assert O.topk_boundary(S, T, 4) == (1.0, None)
    assert O.topk_boundary(S, T, 5) == (None, None)
    # ties: the k-th and (k+1)-th of equal candidates are equal
    St = np.array([0.0, 3, 7, 3, 3, 0])
    assert O.topk_boundary(St, T, 2) == (3.0, 3.0)
    assert O.topk_boundary(St, T, 1) == (7.0, 3.0)
    # no candidates at all (the context ends in block 0 or 1)
    assert O.topk_boundary(S, 64, 1) == (None, None)
    assert O.topk_boundary(S, 65, 1) == (None, None)
    # blocks past the tail are not candidates even if their score is the largest
    assert O.topk_boundary(np.array([0.0, 4, 1, 8, 99, 99]), 3 * 64 + 1, 1) == (4.0, 1.0)


def test_topk_boundary_brackets_the_selection():
    """The k-th value is the smallest chosen candidate score and the (k+1)-th the largest
    unchosen one (by brute force over the selection), and the selection is unique exactly
    when they differ."""
    rng = np.random.default_rng(11)
    for trial in range(300):
        T = int(rng.integers(1, 64 * 30))
        tb = (T - 1) // 64
        S = rng.integers(-3, 4, tb + 3).astype(np.float64)
        k = int(rng.integers(1, 10))
        cand = [j for j in range(tb + 1) if j not in (0, tb)]
        chosen = [j for j in _brute_select(S, T, k) if j not in (0, tb)]
        left = [j for j in cand if j not in chosen]
        kth, k1 = O.topk_boundary(S, T, k)
        if k <= len(cand):
            assert kth == min(S[j] for j in chosen)
        else:
            assert kth is None
        if left and k < len(cand):
            assert k1 == max(S[j] for j in left)
        else:
            assert k1 is None


# ---------------------------------------------------------------- baseline selector
def test_multihead_scores_closed_form():
    ck = np.array([[1.0, 0.0], [0.0, 0.0]])
    q = np.array([[math.sqrt(2) * math.log(3), 0.0], [0.0, 0.0]])
    # head 0: logits ln3, 0 -> (3/4, 1/4); head 1: uniform (1/2, 1/2)
    assert np.allclose(O.multihead_scores(q, ck), [1.25, 0.75], rtol=0, atol=1e-15)


def test_single_head_forecast_equals_multihead_with_identical_queries():
    # A sum of identical per-head softmaxes is a monotone map of one head's scores, so the
    # 16-head softmax-summed selector picks the same blocks as the single forecast head.
    rng = np.random.default_rng(4)
    for trial in range(4):
        T = 4096
        K = O.bf16_round(rng.standard_normal((T, 128)))
        f = O.bf16_round(rng.standard_normal(128))
        W = O.num_windows(T - 1)
        ck = O.compress_keys(K, W)
        nb = (T - 1) // 64 + 1
        S1 = O.pool_to_blocks(O.forecast_scores(ck, f), nb)
        S16 = O.pool_to_blocks(O.multihead_scores(np.tile(f, (16, 1)), ck), nb)
        assert O.select_blocks(S1, T, 8) == O.select_blocks(S16, T, 8)


def test_forecast_scale_invariance():
    rng = np.random.default_rng(5)
    T = 2048
    K = O.bf16_round(rng.standard_normal((T, 16)))
    f = rng.standard_normal(16)
    sel = O.forecast_select_one(K, f, T, 5)
    assert O.forecast_select_one(K, 3.0 * f, T, 5) == sel
    # Negating f negates every window score, so the block score becomes minus the LOWEST
    # window score over the block: the selection turns into the 5 blocks whose lowest
    # overlapping window score is smallest (windows 4j-1 .. 4j+3 overlap block j).
    W = O.num_windows(T - 1)
    s = O.compress_keys(K, W) @ f
    tb = (T - 1) // 64
    lowest = {j: min(s[max(0, 4 * j - 1):min(W, 4 * j + 4)]) for j in range(1, tb)}
    bottom = sorted(lowest, key=lambda j: (lowest[j], j))[:5]
    assert O.forecast_select_one(K, -f, T, 5) == sorted({0, tb} | set(bottom))


# ---------------------------------------------------------------- attention
def test_sparse_attention_with_all_blocks_equals_dense():
    rng = np.random.default_rng(6)
    for T in (1, 63, 64, 65, 700):
        K = rng.standard_normal((T + 5, 32))
        V = rng.standard_normal((T + 5, 32))
        q = rng.standard_normal((16, 32))
        sel = list(range((T - 1) // 64 + 1))
        a = O.block_sparse_attention(q, K, V, sel, T)
        b = O.dense_causal_attention(q, K, V, T)
        assert np.allclose(a, b, rtol=1e-12, atol=1e-12)


def test_attention_single_token_returns_its_value():
    rng = np.random.default_rng(7)
    K = rng.standard_normal((10, 8))
    V = rng.standard_normal((10, 8))
    q = rng.standard_normal((4, 8))
    out = O.block_sparse_attention(q, K, V, [0], 1)
    assert np.allclose(out, np.tile(V[0], (4, 1)), rtol=0, atol=1e-15)


def test_attention_ignores_selection_order_and_masks_future_tokens():
    rng = np.random.default_rng(8)
    T = 300
    K = rng.standard_normal((320, 16))
    V = rng.standard_normal((320, 16))
    q = rng.standard_normal((3, 16))
    a = O.block_sparse_attention(q, K, V, [0, 2, 4], T)
    b = O.block_sparse_attention(q, K, V, [4, 0, 2], T)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-13)
    V2 = V.copy()
    V2[T:] = 1e6                                             # beyond the context
    assert np.allclose(O.block_sparse_attention(q, K, V2, [0, 2, 4], T), a, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- forecast projection
def test_forecast_project_small_integers_and_rounding():
    W = np.array([[1.0, 2, 3], [4, 5, 6]])
    h = np.array([1.0, -1, 2])
    assert np.array_equal(O.forecast_project(W, h), [5, 11])
    e = 2.0 ** -8
    assert O.forecast_project(np.array([[1.0, e]]), np.array([1.0, 1.0]))[0] == 1.0
    assert O.forecast_project(np.array([[1.0, 1.5 * e]]), np.array([1.0, 1.0]))[0] == 1 + 2 * e


# ---------------------------------------------------------------- golden hand case
def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            vals[key] = val.split()
    return vals


def _num(tok):
    if tok == "-inf":
        return -np.inf
    if tok == "sqrt2ln3":
        return math.sqrt(2) * math.log(3)
    if "/" in tok:
        a, b = tok.split("/")
        return float(a) / float(b)
    return float(tok)


def test_golden_hand_decode_case():
    g = _read_golden("hand_decode_case.txt")
    T = 200
    K = np.zeros((256, 2))
    K[64:128] = (1, 0)
    K[128:192] = (0, 2)
    V = np.stack([np.arange(256, dtype=np.float64), np.ones(256)], axis=1)
    f = np.array([3.0, 1.0])
    W = O.num_windows(T - 1)
    ck = O.compress_keys(K, W)
    s = O.forecast_scores(ck, f)
    assert np.array_equal(s, [_num(t) for t in g["window_scores"]])
    S = O.pool_to_blocks(s, 4)
    assert np.array_equal(S, [_num(t) for t in g["block_scores"]])
    sel = O.forecast_select_one(K, f, T, 1)
    assert sel == [int(t) for t in g["selected"]]
    q = np.array([[_num(t) for t in g["q_head_a"]], [_num(t) for t in g["q_head_b"]]])
    out = O.block_sparse_attention(q, K, V, sel, T)
    want = np.array([[_num(t) for t in g["out_head_a"]], [_num(t) for t in g["out_head_b"]]])
    assert np.allclose(out, want, rtol=1e-13, atol=0)


# ---------------------------------------------------------------- readings
def test_window_ending_at_current_token_is_not_scored():
    # T = 208: the window 176..207 ends at the current token 207, so under lookahead it does
    # not exist yet for the target layer. Huge keys in 192..207 would lift block 2 through
    # that window (it overlaps block 2) if it were scored.
    T = 208
    K = np.zeros((256, 2))
    K[64:128] = (1, 0)              # block 1 moderately aligned with f
    K[192:208] = (100, 0)           # only window 11 (176..207) reaches these
    f = np.array([1.0, 0.0])
    assert O.forecast_select_one(K, f, T, 1) == [0, 1, 3]


def test_decode_step_lookahead_wiring():
    # Three layers, one group, d = 4, hidden = 4. Layer 0's self head and each layer's next
    # head produce a distinct unit forecast; each layer's keys hold one block aligned with
    # exactly the forecast meant to select it, so a lookahead wired to the wrong layer or
    # head picks a different block.
    d, hidden, B, G, H = 4, 4, 1, 1, 2
    T_cap, p = 8 * 64, 8 * 64 - 1
    eye = np.eye(4)
    W_self0 = eye[[0, 1, 2, 3]]      # f = h
    W_next = [eye[[1, 2, 3, 0]], eye[[2, 3, 1, 0]]]
    h = [eye[[0]], eye[[1]], eye[[2]]]               # a distinct hidden state per layer
    # forecasts: layer 0 self: e0; layer 1 (layer 0's next head on h0): e3; layer 2 (layer
    # 1's next head on h1): e2. Any other head/hidden pairing gives e0, e1 or e3 instead.
    f_self0 = W_self0 @ h[0][0]
    f_l1 = W_next[0] @ h[0][0]
    f_l2 = W_next[1] @ h[1][0]
    layers = []
    target = {0: (f_self0, 1), 1: (f_l1, 3), 2: (f_l2, 5)}
    for L in range(3):
        K = np.zeros((B, G, T_cap, d))
        V = np.zeros((B, G, T_cap, d))
        fv, blk = target[L]
        K[0, 0, blk * 64:(blk + 1) * 64] = 4 * fv
        # a decoy block aligned with every other layer's forecast
        for L2, (fv2, blk2) in target.items():
            if L2 != L and not np.allclose(fv2, fv):
                K[0, 0, (blk2 + 1) * 64:(blk2 + 2) * 64] = 4 * fv2
        layers.append((K, V))
    q = [np.zeros((B, G * H, d))] * 3
    kv0 = [np.zeros((B, G, d))] * 3
    sel, out = O.decode_step(layers, W_self0, W_next, h, q, kv0, kv0, p, 1, H)
    assert sel[0][0][0] == [0, 1, 7]
    assert sel[1][0][0] == [0, 3, 7]
    assert sel[2][0][0] == [0, 5, 7]


def test_decode_step_first_token_attends_itself():
    d, hidden, B, G, H = 8, 4, 2, 2, 3
    rng = np.random.default_rng(9)
    layers = [(np.zeros((B, G, 64, d)), np.zeros((B, G, 64, d))) for _ in range(2)]
    W_self0 = rng.standard_normal((G * d, hidden))
    W_next = [rng.standard_normal((G * d, hidden))]
    h = [rng.standard_normal((B, hidden)) for _ in range(2)]
    q = [rng.standard_normal((B, G * H, d)) for _ in range(2)]
    kn = [rng.standard_normal((B, G, d)) for _ in range(2)]
    vn = [rng.standard_normal((B, G, d)) for _ in range(2)]
    sel, out = O.decode_step(layers, W_self0, W_next, h, q, kn, vn, 0, 4, H)
    for L in range(2):
        for b in range(B):
            for g in range(G):
                assert sel[L][b][g] == [0]
                assert np.allclose(out[L][b, g * H:(g + 1) * H], vn[L][b, g], atol=1e-15)


# ---------------------------------------------------------------- prefill (chunked queries)
def _brute_attention(q_heads, K, V, toks, scale):
    """Softmax attention of each head over an explicit token list, by a plain loop."""
    out = np.zeros((q_heads.shape[0], V.shape[1]))
    for h in range(q_heads.shape[0]):
        logits = [float(q_heads[h] @ K[t]) * scale for t in toks]
        m = max(logits)
        w = [math.exp(x - m) for x in logits]
        tot = sum(w)
        for wi, t in zip(w, toks):
            out[h] += wi / tot * V[t]
    return out


def test_prefill_chunk_windows_are_those_before_the_chunk():
    for c in range(0, 40):
        brute = sum(1 for i in range(0, 400) if 16 * i + 32 <= 64 * c)
        assert O.prefill_chunk_windows(c) == brute
    assert [O.prefill_chunk_windows(c) for c in range(4)] == [0, 3, 7, 11]
    assert O.prefill_num_chunks(1) == 1 and O.prefill_num_chunks(64) == 1 and O.prefill_num_chunks(65) == 2


def test_prefill_forecast_scores_small_integers():
    rng = np.random.default_rng(21)
    ck = rng.integers(-3, 4, (20, 4)).astype(np.float64)
    F = rng.integers(-2, 3, (5, 4)).astype(np.float64)
    c = 3                                                   # windows 0 .. 10 exist before chunk 3
    s = O.prefill_forecast_scores(F, ck, c)
    assert s.shape == (11,)
    for i in range(11):
        assert s[i] == sum(sum(F[t, e] * ck[i, e] for e in range(4)) for t in range(5))


def test_prefill_window_touching_the_chunk_is_not_scored():
    # a huge compressed key at the first window that overlaps chunk c's own tokens must not
    # change chunk c's selection; one window earlier it must
    rng = np.random.default_rng(22)
    c, d = 6, 8
    ck = rng.normal(size=(40, d))
    f = rng.normal(size=(1, d))
    base = O.prefill_select(O.pool_to_blocks(O.prefill_forecast_scores(f, ck, c), c + 1), c, 1)
    W = O.prefill_chunk_windows(c)
    hot = ck.copy()
    hot[W] = 100 * f[0]
    assert O.prefill_select(O.pool_to_blocks(O.prefill_forecast_scores(f, hot, c), c + 1), c, 1) == base
    hot = ck.copy()
    hot[W - 2] = 100 * f[0]                                 # window 4c-3 lies in block c-1 only
    assert O.prefill_select(O.pool_to_blocks(O.prefill_forecast_scores(f, hot, c), c + 1), c, 1) == [0, c - 1, c]


def test_prefill_constant_forecast_equals_the_decode_selection():
    """A chunk whose tokens all carry the same forecast selects what a decode step with that
    forecast selects when its current token is the first token of the chunk's block (the
    decode step scores the windows before its current token, and its tail block is c)."""
    rng = np.random.default_rng(23)
    T, d, k = 64 * 9 + 17, 16, 3
    K = rng.normal(size=(T, d))
    ck = O.compress_keys(K, O.num_windows(T))
    for c in range(O.prefill_num_chunks(T)):
        f = rng.normal(size=d)
        n_tok = min(64, T - 64 * c)
        sc = O.prefill_forecast_scores(np.tile(f, (n_tok, 1)), ck, c)
        got = O.prefill_select(O.pool_to_blocks(sc, c + 1), c, k)
        assert got == O.forecast_select_one(K, f, 64 * c + 1, k)
        # positive per-token weights sum to a positive multiple: the same selection
        w = rng.uniform(0.5, 2.0, size=(n_tok, 1))
        sw = O.prefill_forecast_scores(w * f, ck, c)
        assert O.prefill_select(O.pool_to_blocks(sw, c + 1), c, k) == got
    assert O.prefill_select(np.zeros(1), 0, 4) == [0]
    assert O.prefill_select(np.zeros(2), 1, 4) == [0, 1]


def test_prefill_multihead_with_identical_queries_equals_forecast():
    rng = np.random.default_rng(24)
    T, d, H, k = 64 * 7, 8, 4, 2
    K = rng.normal(size=(T, d))
    ck = O.compress_keys(K, O.num_windows(T))
    for c in range(2, 7):
        qv = rng.normal(size=d)
        Qc = np.tile(qv, (64, H, 1))
        mh = O.pool_to_blocks(O.prefill_multihead_scores(Qc, ck, c), c + 1)
        fc = O.pool_to_blocks(O.prefill_forecast_scores(np.tile(qv, (64, 1)), ck, c), c + 1)
        assert O.prefill_select(mh, c, k) == O.prefill_select(fc, c, k)
        # the sum of 64 x H identical softmaxes is 64 H times one softmax
        s1 = O.multihead_scores(qv[None, :], ck[:O.prefill_chunk_windows(c)])
        assert np.allclose(O.prefill_multihead_scores(Qc, ck, c), 64 * H * s1, rtol=1e-12)


def test_prefill_attention_with_all_blocks_equals_dense_causal():
    rng = np.random.default_rng(25)
    T, H, d = 64 * 3 + 21, 3, 8
    Q, K, V = rng.normal(size=(T, H, d)), rng.normal(size=(T, d)), rng.normal(size=(T, d))
    n = O.prefill_num_chunks(T)
    sel = [O.prefill_select(rng.normal(size=c + 1), c, 99) for c in range(n)]
    assert sel[-1] == list(range(n))
    got = O.prefill_block_sparse_attention(Q, K, V, sel, T)
    assert np.allclose(got, O.dense_causal_prefill_attention(Q, K, V, T), rtol=1e-12, atol=1e-12)
    assert np.allclose(got[0], np.tile(V[0], (H, 1)))        # the first token attends itself only


def test_prefill_attention_is_causal_within_the_selected_blocks():
    rng = np.random.default_rng(26)
    T, H, d = 64 * 5 + 9, 2, 8
    Q, K, V = rng.normal(size=(T, H, d)), rng.normal(size=(T, d)), rng.normal(size=(T, d))
    sel = [[0], [0, 1], [0, 2], [0, 1, 3], [0, 2, 4], [0, 3, 5]]
    got = O.prefill_block_sparse_attention(Q, K, V, sel, T)
    scale = 1 / math.sqrt(d)
    for t in [0, 5, 63, 64, 100, 130, 191, 192, 250, 256, 300, T - 1]:
        toks = [u for u in range(t + 1) if u // 64 in sel[t // 64]]
        assert np.allclose(got[t], _brute_attention(Q[t], K, V, toks, scale), rtol=1e-12, atol=1e-12)
    # a future token inside the chunk's own block changes nothing before it
    V2 = V.copy()
    V2[64 * 4 + 30] += 10.0
    got2 = O.prefill_block_sparse_attention(Q, K, V2, sel, T)
    assert np.array_equal(got2[:64 * 4 + 30], got[:64 * 4 + 30])
    assert not np.allclose(got2[64 * 4 + 30], got[64 * 4 + 30])
