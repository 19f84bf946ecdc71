"""Block index keys (oracle; test-only).

The pages score KV *blocks* ("attention scoring -> per-block importance", OasisKV page,
key module 2) but do not say how a block is summarised.  Reading used here: the index key
of block b is the mean of its present keys,

    ik[b] = bf16_rne( (sum over t in block b, t < L, ascending, of fp32(k_t)) / n_b )

with the sum taken in fp32 one token at a time in ascending position, an IEEE fp32
division by the number n_b of present tokens, and bf16 round-to-nearest-even.  By
linearity q.ik[b] is the mean token logit of the block, at 1/bs of the key bytes, so the
scoring keys stay on the GPU while the full K/V lives in host memory (HiSparse page,
insight 1: GPU footprint bounded).  With block size 1, ik is the key itself.

Pinned by tests/test_oracle_index_keys.py: a hand-computed partial-block fixture
(tests/golden/index_keys_small.json), bs = 1 identity, and exact-mean cases.
"""
import numpy as np

from .bf16 import bf16_to_f32, f32_to_bf16_rne


def _f32(rows: np.ndarray) -> np.ndarray:
    """Key rows as fp32 values: bf16 bit patterns (uint16) are widened; fp32 values (dequantized
    FP8 keys) are taken as they are."""
    return rows if rows.dtype == np.float32 else bf16_to_f32(rows)


def index_key_block(k_rows: np.ndarray) -> np.ndarray:
    """Index key of one block from its present key rows (n_b, D): bf16 bit patterns or fp32 values."""
    n = k_rows.shape[0]
    if n == 0:
        raise ValueError("a block with no present token has no index key")
    acc = np.zeros(k_rows.shape[1], np.float32)
    for t in range(n):                       # ascending token order, fp32 adds
        acc = acc + _f32(k_rows[t])
    mean = acc / np.float32(n)               # IEEE fp32 division
    return f32_to_bf16_rne(mean)


def index_keys(k_rows: np.ndarray, ctx_len: int, block_size: int) -> np.ndarray:
    """Index keys of blocks 0 .. ceil(ctx_len / bs) - 1 of one (request, layer, kv-head).

    k_rows: (>= ctx_len, D) bf16 bit patterns; returns (n_blocks, D) bf16 bit patterns.
    Vectorised over blocks; per block the sum still runs token by token in order."""
    nb = (ctx_len + block_size - 1) // block_size
    d = k_rows.shape[1]
    out = np.empty((nb, d), np.uint16)
    n_full = ctx_len // block_size
    if n_full:
        blocks = _f32(k_rows[: n_full * block_size]).reshape(n_full, block_size, d)
        acc = np.zeros((n_full, d), np.float32)
        for t in range(block_size):
            acc = acc + blocks[:, t, :]
        out[:n_full] = f32_to_bf16_rne(acc / np.float32(block_size))
    if nb > n_full:
        out[n_full] = index_key_block(k_rows[n_full * block_size: ctx_len])
    return out
