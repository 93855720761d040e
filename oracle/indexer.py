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

from . import formats


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


def scores_fp8(q_codes: np.ndarray, w: np.ndarray, key_codes: np.ndarray, key_scales: np.ndarray) -> np.ndarray:
    """FP8 keys as on the pages ("vLLM Part 2", footnote 3: 128 FP8 values plus a
    4-byte scale per key).

    q_codes [H_i, 128] e4m3 codes, w [H_i] fp32 head weights (the query's own scale
    folded in, any sign), key_codes [n, 128] e4m3 codes, key_scales [n] fp32
    -> [n] fp64:  s[t] = scale_t * sum_h w_h * max(0, sum_d q[h, d] * k_t[d]).
    Reading: the scale multiplies the dequantised key; key scales are amax / 448 of
    the key (never negative), so the scale may stand outside the ReLU."""
    q = formats.e4m3_to_f64(np.asarray(q_codes, np.uint8))
    k = formats.e4m3_to_f64(np.asarray(key_codes, np.uint8))
    d = k @ q.T                                                       # [n, H_i]
    return np.asarray(key_scales, np.float64) * (np.maximum(d, 0.0) @ np.asarray(w, np.float64))


def topk_real(s: np.ndarray, k: int) -> np.ndarray:
    """topk for real-valued scores: (-score, token) ascending, the same rule."""
    n = len(s)
    order = np.lexsort((np.arange(n), -np.asarray(s, np.float64)))
    sel = np.sort(order[:min(k, n)])
    out = np.full(k, -1, np.int32)
    out[:len(sel)] = sel
    return out
