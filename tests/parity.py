"""Comparison rules of the parity tests (CUDA path vs the fp64 oracle).

Selected blocks: integer output decided by floating point. The CUDA selector scores in
float32 and the oracle in float64, so at a near-tie of the k-th and (k+1)-th candidate
block scores both selections are correct. The rule: where the oracle's k-th and (k+1)-th
candidate scores differ by more than 1e-4 relative, the selection is unique and must match
bit for bit; otherwise every block whose oracle score is clearly above the k-th (by more than
the band) must be selected, none clearly below it may be, and the count must be right. The
forced blocks, ascending order and -1 padding are always checked exactly.

Attention: max |gpu - oracle| <= 1e-2 * max |oracle| + 2e-3 per (sequence, group), for bf16
inputs with float32 accumulation.
"""
import numpy as np

from oracle import sparda_oracle as O

REL_GAP = 1e-4


def to64(t):
    return t.detach().double().cpu().numpy()


def check_selection(idx_row, cnt, S, T, k):
    """Checks one (sequence, group) selection against the oracle's block scores S.

    Returns True when the selection was unique (compared bit for bit), False when it sat in
    a near-tie band (compared by validity)."""
    idx_row = [int(x) for x in idx_row]
    cnt = int(cnt)
    tb = (T - 1) // 64
    forced = {0, tb}
    cand = [j for j in range(tb + 1) if j not in forced]
    k_eff = min(k, len(cand))
    assert cnt == k_eff + len(forced), (cnt, k_eff, forced)
    sel = idx_row[:cnt]
    assert all(x == -1 for x in idx_row[cnt:]), idx_row
    assert sel == sorted(set(sel)), sel
    assert forced <= set(sel)
    chosen = set(sel) - forced
    assert chosen <= set(cand) and len(chosen) == k_eff
    want = O.select_blocks(S, T, k)
    if k_eff == 0 or k_eff == len(cand):
        assert sel == want
        return True
    kth, k1 = O.topk_boundary(S, T, k)
    band = REL_GAP * max(abs(kth), abs(k1))
    if kth - k1 > band:
        assert sel == want, ("unique selection differs", sel, want)
        return True
    for j in cand:
        if S[j] > kth + band:
            assert j in chosen, ("clearly-in block missing", j)
        if S[j] < kth - band:
            assert j not in chosen, ("clearly-out block chosen", j)
    return False


def attn_tol(o_ref):
    return 1e-2 * float(np.max(np.abs(o_ref))) + 2e-3


def check_attention(o_gpu, o_ref):
    err = float(np.max(np.abs(o_gpu - o_ref)))
    tol = attn_tol(o_ref)
    assert err <= tol, ("attention error", err, tol)
    return err
