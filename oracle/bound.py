"""Block min/max summaries and the query-aware upper-bound block score (oracle; test-only).

A second block-scoring mode beside the block-mean key.  The pages name Quest among the top-k
selector families a host-KV cache serves (HiSparse page, insights 1 and 3; "大模型推理加速" page:
in decode Quest generalises best because it uses the query to choose the KV), without its formula;
this restates the published Quest rule (Tang et al., 2024) in the terms used here:

    mx[b][d] = max over present tokens t of block b of k_t[d]      (bf16: no rounding)
    mn[b][d] = min over the same tokens
    s[b]     = scale * max over scoring rows r of  sum_d max(q_r[d] * mx[b][d], q_r[d] * mn[b][d])

which is the largest logit any key inside the block's per-channel box could give, hence an upper
bound of the block's largest token logit (and equal to it for a one-token block).  The stored
summary row is [mx | mn] (2 * d_k wide).  Sums in fp64 (every bf16 x bf16 product is exact in
fp64); A[b] = scale * max_r sum_d |term_d| is the conditioning used by the score tolerance.

Pinned by tests/test_oracle_bound.py: a hand-worked fixture (tests/golden/bound_small.json), the
upper-bound property against brute force over the tokens, equality on one-token blocks, and the
summary of a one-token block being [k | k].
"""
import numpy as np

from .bf16 import bf16_to_f32, bf16_to_f64


def index_minmax_block(k_rows: np.ndarray) -> np.ndarray:
    """[max | min] over the present rows (n, D) of one block, bf16 patterns -> (2 D,) patterns."""
    if k_rows.shape[0] == 0:
        raise ValueError("a block with no present token has no summary")
    vals = bf16_to_f32(k_rows)
    hi = np.argmax(vals, axis=0)
    lo = np.argmin(vals, axis=0)
    cols = np.arange(k_rows.shape[1])
    return np.concatenate([k_rows[hi, cols], k_rows[lo, cols]]).astype(np.uint16)


def index_minmax(k_rows: np.ndarray, ctx_len: int, block_size: int) -> np.ndarray:
    """[max | min] summaries of blocks 0 .. ceil(ctx_len / bs) - 1: (n_blocks, 2 D) bf16 patterns."""
    nb = (ctx_len + block_size - 1) // block_size
    out = np.empty((nb, 2 * k_rows.shape[1]), np.uint16)
    for b in range(nb):
        out[b] = index_minmax_block(k_rows[b * block_size: min(ctx_len, (b + 1) * block_size)])
    return out


def block_scores_bound(q_rows: np.ndarray, summ: np.ndarray, scale: float):
    """q_rows (R, D) bf16 patterns; summ (n_blocks, 2 D) [max | min] -> (s, A) fp64 (n_blocks,)."""
    d = q_rows.shape[1]
    q = bf16_to_f64(q_rows)                      # (R, D)
    mx = bf16_to_f64(summ[:, :d])                # (n, D)
    mn = bf16_to_f64(summ[:, d:])
    t_hi = q[:, None, :] * mx[None, :, :]        # (R, n, D)
    t_lo = q[:, None, :] * mn[None, :, :]
    terms = np.maximum(t_hi, t_lo)
    s = float(scale) * terms.sum(axis=2).max(axis=0)
    a = float(scale) * np.abs(terms).sum(axis=2).max(axis=0)
    return s, a
