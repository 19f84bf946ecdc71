"""Exact decode attention over a token set (oracle; test-only).

    o_h = sum_t softmax_t(scale * q_h . k_t) v_t      for each q head h of the group

over the tokens t of the selected blocks with t < L, in ascending position, in fp64 with
the maximum logit subtracted before exp; the result is rounded to fp32.  Sparse attention
over the HBM-resident selection is exact attention over those tokens (OasisKV page, key
module 1: exact foreground attention over the sparse KV in HBM; HiSparse page, insight 1:
outputs identical to full KV in HBM), so the oracle is the plain definition.  With no
token the output is zero.  MLA reading: K is the full latent row, V its first d_v entries.

Pinned by tests/test_oracle_attention.py: torch's scaled_dot_product_attention in fp64 (a
library routine), one token -> v, equal logits -> mean of v, and a budget >= context giving
dense attention.
"""
import numpy as np

from .bf16 import bf16_to_f64


def attend(q_rows: np.ndarray, k_tok: np.ndarray, v_tok: np.ndarray, scale: float) -> np.ndarray:
    """q_rows (G, D_k) bf16 patterns; k_tok (T, D_k), v_tok (T, D_v): bf16 patterns or float64
    values (dequantized FP8 rows) -> (G, D_v) fp32."""
    g, dv = q_rows.shape[0], v_tok.shape[1]
    if k_tok.shape[0] == 0:
        return np.zeros((g, dv), np.float32)

    def f64(a):
        return a if a.dtype == np.float64 else bf16_to_f64(a)

    q, k, v = bf16_to_f64(q_rows), f64(k_tok), f64(v_tok)
    logits = float(scale) * (q @ k.T)
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    o = (p @ v) / p.sum(axis=1, keepdims=True)
    return o.astype(np.float32)
