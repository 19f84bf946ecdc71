"""Block scores (oracle; test-only).

    s[b] = scale * max_{r in scoring rows} ( q_r . ik[b] )

The scoring rows of one (request, kv-head) are the q heads of its GQA group (q head h
belongs to kv head floor(h / G)), for each scoring query: the current query in sync mode, or
each lookahead draft in lookahead mode.  Sources: tuntang.top survey, section 3 step 3 (take
an element-wise max of attention scores within a GQA group before choosing top-K per group);
OasisKV page, key module 2 (draft lookahead tokens score every KV block); "attention score"
is S = Q.K^T (KV-cache overview, section 3.1).

The dot products are accumulated in fp64 (bf16 x bf16 products are exact in fp64), and
the caller rounds s to fp32 for selection.  A[b] = scale * max_r sum_d |q_r,d * ik[b],d|
is returned too: it bounds the conditioning of s[b], and the GPU tolerance is
|s_gpu - s| <= 1e-4 (|s| + A).

Pinned by tests/test_oracle_scores.py: exactly-rounded sums (math.fsum) on small inputs,
the single-row/single-head reduction to a dot product, and the group-max rule.
"""
import numpy as np

from .bf16 import bf16_to_f64


def block_scores(q_rows: np.ndarray, ik: np.ndarray, scale: float):
    """q_rows: (R, D) bf16 patterns; ik: (n_blocks, D) bf16 patterns -> (s, A) fp64 (n_blocks,)."""
    q = bf16_to_f64(q_rows)
    k = bf16_to_f64(ik)
    dots = q @ k.T                                   # (R, n_blocks)
    s = float(scale) * dots.max(axis=0)
    a = float(scale) * (np.abs(q) @ np.abs(k).T).max(axis=0)
    return s, a
