"""Pins for oracle.bf16: hand-derived rounding cases and torch's float32 -> bfloat16 conversion."""
import numpy as np
import pytest
import torch

from oracle import bf16_to_f32, f32_to_bf16_rne


def _bits(x):
    return np.array([x], np.float32).view(np.uint32)[0]


@pytest.mark.parametrize("f32_bits, bf16_bits", [
    (0x3F800000, 0x3F80),  # 1.0 exact
    (0x3F808000, 0x3F80),  # 1 + 2^-8: tie, kept fraction even -> down
    (0x3F818000, 0x3F82),  # 1 + 3*2^-8: tie, kept fraction odd -> up
    (0x3F808001, 0x3F81),  # just above half -> up
    (0x3F807FFF, 0x3F80),  # just below half -> down
    (0x3FFF8000, 0x4000),  # tie with odd fraction 0x7F: carry into the exponent (2.0)
    (0x7F7FFFFF, 0x7F80),  # max float rounds to +inf
    (0xFF7FFFFF, 0xFF80),  # -max -> -inf
    (0x80000000, 0x8000),  # -0.0 keeps its sign
    (0x00000001, 0x0000),  # smallest subnormal rounds to +0
    (0x7F800000, 0x7F80),  # +inf
])
def test_hand_cases(f32_bits, bf16_bits):
    x = np.array([f32_bits], np.uint32).view(np.float32)
    assert int(f32_to_bf16_rne(x)[0]) == bf16_bits


def test_nan_stays_nan():
    x = np.array([0x7FC00001, 0xFF800001], np.uint32).view(np.float32)
    out = f32_to_bf16_rne(x)
    assert np.isnan(bf16_to_f32(out)).all()
    assert int(out[1]) & 0x8000


def test_matches_torch_on_random_and_edges():
    rng = np.random.default_rng(0)
    u = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    x = x[~np.isnan(x)]
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(f32_to_bf16_rne(x), ref)


def test_widening_is_exact():
    b = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    f = bf16_to_f32(b)
    ok = ~np.isnan(f)
    ref = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(f[ok], ref[ok])
    np.testing.assert_array_equal(f32_to_bf16_rne(f[ok]), b[ok])
