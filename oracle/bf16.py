"""bf16 <-> binary32 conversions written from the IEEE-754 definitions (oracle; test-only).

bfloat16 keeps the sign, the 8 exponent bits and the top 7 fraction bits of binary32.
Rounding to nearest, ties to even: drop the low 16 bits of the binary32 pattern; round up
when the dropped part is above half an ulp, or exactly half with an odd kept part.  A
carry out of the fraction increments the exponent, which is the correct next value
(including overflow to infinity).  NaN inputs map to a quiet NaN of the same sign.

Pinned by tests/test_oracle_bf16.py: hand-derived tie and carry cases and torch's CPU
float32 -> bfloat16 conversion (a library routine) on random and edge values.
"""
import numpy as np


def f32_to_bf16_rne(x) -> np.ndarray:
    u = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)
    kept = u >> np.uint32(16)
    dropped = u & np.uint32(0xFFFF)
    half = np.uint32(0x8000)
    round_up = (dropped > half) | ((dropped == half) & ((kept & np.uint32(1)) == np.uint32(1)))
    out = kept + round_up.astype(np.uint32)
    is_nan = (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    out = np.where(is_nan, (kept & np.uint32(0x8000)) | np.uint32(0x7FC0), out)
    return out.astype(np.uint16)


def bf16_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_to_f64(b) -> np.ndarray:
    return bf16_to_f32(b).astype(np.float64)
