"""Comparison rules between the CUDA path and the oracle.

Top-K: indices must equal the oracle's bit for bit, except where the oracle's
K-th and (K+1)-th scores differ by less than 1e-5 relative; there every
position the two sets disagree on must score within that band of the K-th
score.  Attention: max-abs error <= 2e-3 for bf16 inputs with fp32
accumulation, <= 1e-5 for the fp32 configuration, computed by the oracle on
the GPU's own index set.
"""
import numpy as np

TOPK_REL = 1e-5
ATOL_BF16 = 2e-3
ATOL_F32 = 1e-5


def check_topk_row(g, o, scores, pos, K, rel=TOPK_REL):
    """Return the number of tie-band swaps (0 = identical); assert on failure."""
    n = min(K, pos + 1)
    g = np.asarray(g)
    assert (g[n:] == -1).all(), "padding must be -1"
    gs = g[:n]
    assert (gs >= 0).all() and (gs <= pos).all(), "index outside 0..pos"
    assert (np.diff(gs) > 0).all(), "indices must be strictly ascending"
    os_ = np.asarray(o)[:n]
    if np.array_equal(gs, os_):
        return 0
    sc = np.asarray(scores, dtype=np.float64)[: pos + 1]
    srt = np.sort(sc)[::-1]
    th_k, th_k1 = srt[K - 1], srt[K]
    band = rel * abs(th_k)
    assert th_k - th_k1 < band, f"differs although K-th/K+1-th gap {th_k - th_k1} >= {band}"
    diff = np.setxor1d(gs, os_)
    assert (np.abs(sc[diff] - th_k) <= band).all(), "swapped positions outside the tie band"
    return len(diff) // 2


def check_topk(g_idx, o_idx, o_scores, q_pos, K, rows=None):
    rows = range(len(g_idx)) if rows is None else rows
    swaps = 0
    for i, r in enumerate(rows):
        swaps += check_topk_row(g_idx[i], o_idx[i], o_scores[i], int(q_pos[r]), K)
    return swaps


def max_abs(a, b):
    return float(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64)).max())
