"""FP8 E4M3 encode / decode written from the format's definition (oracle; test-only).

The KV-cache overview (section 3.2) names FP8 E4M3 (3 mantissa bits) as the 8-bit format that
keeps the KV cache's accuracy while halving its bytes.  E4M3 as used here (the "fn" variant): a
sign bit, 4 exponent bits with bias 7 and 3 mantissa bits; exponent field e in 1..15 gives
(1 + m/8) * 2^(e-7), e = 0 gives the subnormals m * 2^-9, and S.1111.111 is NaN, so the largest
finite magnitude is 1.75 * 2^8 = 448 and there is no infinity.

Encoding a real x (the quantisation of a stored key or value, x = value / scale in fp32): round to
the nearest representable magnitude, ties to the even mantissa; magnitudes beyond 448 (and
infinities) saturate to 448 ("satfinite"); NaN encodes as 0x7F.  A stored value is then
decode(code) * scale.

Pinned by tests/test_oracle_fp8.py: hand-worked codes (tests/golden/fp8_e4m3.json) including
ties, subnormals and saturation, every one of the 256 codes decoded against torch's float8_e4m3fn
(a library routine), and random in-range values encoded against torch's cast.
"""
import math

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """uint8 codes -> float64 values (NaN for the two NaN codes)."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((e == 15) & ((c & 0x7) == 7), np.nan, val)
    return s * val


def _encode_one(x: float) -> int:
    if x != x:
        return 0x7F
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    if a >= E4M3_MAX:
        return sign | 0x7E
    if a < 2.0 ** -6:                                  # subnormal grid, spacing 2^-9
        q = a / 2.0 ** -9
        m = math.floor(q)
        r = q - m
        if r > 0.5 or (r == 0.5 and m % 2 == 1):
            m += 1
        if m == 8:                                      # rounded up to the smallest normal
            return sign | (1 << 3)
        return sign | m
    mant, exp = math.frexp(a)                           # a = mant * 2^exp, mant in [0.5, 1)
    e = exp - 1                                         # a in [2^e, 2^(e+1))
    q = a / 2.0 ** (e - 3)                              # in [8, 16)
    n = math.floor(q)
    r = q - n
    if r > 0.5 or (r == 0.5 and n % 2 == 1):
        n += 1
    if n == 16:
        n, e = 8, e + 1
    field = e + 7
    if field > 15 or (field == 15 and n - 8 == 7):      # above 448 after rounding: saturate
        return sign | 0x7E
    return sign | (field << 3) | (n - 8)


def e4m3_encode(x) -> np.ndarray:
    """float32 values -> uint8 codes (round to nearest even, saturating to +-448, NaN -> 0x7F).
    The steps of _encode_one, on whole arrays."""
    x32 = np.asarray(x, np.float32)
    a = np.abs(x32.astype(np.float64))
    sign = np.where(np.signbit(x32), 0x80, 0).astype(np.int64)
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        # subnormal grid (a < 2^-6): spacing 2^-9; m == 8 is the smallest normal, whose code is 8 too
        q = a / 2.0 ** -9
        m = np.floor(q)
        r = q - m
        m = m + ((r > 0.5) | ((r == 0.5) & (np.mod(m, 2) == 1)))
        sub_code = m.astype(np.int64)
        # normal grid: a in [2^e, 2^(e+1)), spacing 2^(e-3)
        _, ex = np.frexp(np.where(a > 0, a, 1.0))
        e = ex.astype(np.int64) - 1
        q2 = a / np.exp2(e - 3.0)
        n = np.floor(q2)
        r2 = q2 - n
        n = (n + ((r2 > 0.5) | ((r2 == 0.5) & (np.mod(n, 2) == 1)))).astype(np.int64)
        carry = n == 16
        n = np.where(carry, 8, n)
        e = np.where(carry, e + 1, e)
        field = e + 7
        norm_code = np.where((field > 15) | ((field == 15) & (n - 8 == 7)), 0x7E, (field << 3) | (n - 8))
    code = np.where(a < 2.0 ** -6, sub_code, norm_code)
    code = np.where(a >= E4M3_MAX, 0x7E, code)
    code = sign | code
    code = np.where(np.isnan(a), 0x7F, code)
    return code.astype(np.uint8)


def e4m3_encode_scalar(x: float) -> int:
    """One value through the plain scalar steps (cross-checks the array form)."""
    return _encode_one(float(np.float32(x)))


def quantize(x_bf16_f32, scale: float) -> np.ndarray:
    """Codes of real values stored as fp32 (e.g. bf16 keys widened): encode(fp32(x / scale))."""
    q = (np.asarray(x_bf16_f32, np.float32) / np.float32(scale)).astype(np.float32)
    return e4m3_encode(q)


def dequantize_f32(codes, scale: float) -> np.ndarray:
    """fp32(decode(code) * scale): the stored value, rounded to fp32 as the summaries use it."""
    return (e4m3_decode(codes).astype(np.float32) * np.float32(scale)).astype(np.float32)
