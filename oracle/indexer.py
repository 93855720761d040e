"""Indexer scoring and top-K selection.

Scores follow the lightning-indexer reading adopted for this workload: the pages
("vLLM Part 2", section "Why not TP or DP?") say only that the indexer scores
every earlier token to pick the 2,048 that sparse MLA attends to; the integer
form is s[t] = sum_h w_h * max(0, sum_d q[h, d] * k_t[d]) over int8 q, k, w,
exact in int64. The current token's own key is in the cache, so query token j
sees positions [0, limit_j).

Top-K ("vLLM Part 1", section "Sparsity when you need it": the indexer picks the
top-K tokens): the K largest scores, ties to the lower token index, reported in
ascending token order and padded with -1 when fewer than K tokens exist.
"""
import numpy as np


def scores(q: np.ndarray, w: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """q [H_i, 128] int8, w [H_i] int8, keys [n, 128] int8 -> [n] int64.

    The dot products are integers below 2^24 in magnitude and the weighted sum
    stays below 2^53, so the fp64 matrix product is exact.
    """
    d = np.asarray(keys, np.float64) @ np.asarray(q, np.float64).T      # [n, H_i]
    relu = np.maximum(d, 0.0)
    s = relu @ np.asarray(w, np.float64)
    return np.rint(s).astype(np.int64)


def topk(s: np.ndarray, k: int) -> np.ndarray:
    """Full sort of (-score, token) ascending; first min(k, n) tokens, ascending; -1 pads."""
    n = len(s)
    order = np.lexsort((np.arange(n), -np.asarray(s, np.int64)))
    sel = np.sort(order[:min(k, n)])
    out = np.full(k, -1, np.int32)
    out[:len(sel)] = sel
    return out
