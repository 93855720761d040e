"""Sparse MLA decode attention, MQA form, in fp64.

"vLLM Part 2" footnote on the bytes of a sparse-MLA query: each query reads
2,048 selected 656-byte FP8 KV rows; QK runs over 576 dims and PV over 512.
Every KV row serves all heads (MQA form, section "PCP: split tokens, not heads").
Per head h: z_t = sm_scale * q_h . k_t over the selected rows t (k = the 576
dequantised dims), p = softmax(z), o_h = sum_t p_t v_t with v = the first 512
dims; lse_h = log sum_t exp(z_t). Rows with id -1 are skipped.
"""
import numpy as np

from .formats import dequant_rows, bf16_to_f64

V_DIM = 512


def attend(q_bits: np.ndarray, kv: np.ndarray, sm_scale: float):
    """q_bits [H, 576] bf16 bits; kv [n, 576] float64 -> (o [H, 512], lse [H])."""
    q = bf16_to_f64(q_bits)
    h = q.shape[0]
    if kv.shape[0] == 0:
        return np.zeros((h, V_DIM)), np.full(h, -np.inf)
    z = sm_scale * (q @ kv.T)                     # [H, n]
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    l = e.sum(axis=1, keepdims=True)
    o = (e / l) @ kv[:, :V_DIM]
    lse = (m + np.log(l))[:, 0]
    return o, lse


def sparse_mla_decode(q_bits: np.ndarray, row_ids: np.ndarray, pool_rows: np.ndarray,
                      sm_scale: float):
    """One query token: gather the rows named by row_ids (-1 skipped) from the
    pool ([rows, 656] uint8) and attend over them."""
    ids = np.asarray(row_ids)
    ids = ids[ids >= 0]
    kv = dequant_rows(pool_rows[ids])
    return attend(q_bits, kv, sm_scale)
