"""Pins for oracle.fp8: hand-worked codes (ties, subnormals, saturation), all 256 codes decoded
against torch's float8_e4m3fn, and random in-range values encoded against torch's cast (torch
turns magnitudes above 464 into NaN where this encoder saturates, so the comparison stays within
+-464)."""
import json
import os

import numpy as np
import torch

from conftest import GOLDEN
from oracle.fp8 import dequantize_f32, e4m3_decode, e4m3_encode, e4m3_encode_scalar, quantize


def test_hand_worked_codes():
    with open(os.path.join(GOLDEN, "fp8_e4m3.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        got = int(e4m3_encode(np.array([c["x"]], np.float32))[0])
        assert got == c["code"], (c["x"], got, c["why"])
    assert int(e4m3_encode(np.array([np.nan], np.float32))[0]) == 0x7F
    assert int(e4m3_encode(np.array([np.inf], np.float32))[0]) == 0x7E


def test_decode_every_code_against_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3_decode(codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    np.testing.assert_array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])


def test_encode_against_torch_in_range():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.normal(size=20000) * 4, rng.normal(size=5000) * 100, rng.uniform(-464, 464, 5000),
                        rng.normal(size=5000) * 0.01, np.arange(-464, 465, 0.5)]).astype(np.float32)
    x = x[np.abs(x) <= 464.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(e4m3_encode(x), ref)


def test_round_trip_and_scale():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    np.testing.assert_array_equal(e4m3_encode(e4m3_decode(codes).astype(np.float32)), np.where(codes == 0x80, 0x80, codes))
    x = np.array([1.0, -3.0, 0.25], np.float32)
    np.testing.assert_array_equal(dequantize_f32(quantize(x, 0.5), 0.5), x)


def test_array_encoder_matches_the_scalar_steps():
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.normal(size=3000) * 50, rng.normal(size=2000) * 0.003, [0.0, -0.0, 1e-30, 5e5, -np.inf],
                        np.arange(0, 2 ** -5, 2 ** -12)]).astype(np.float32)
    np.testing.assert_array_equal(e4m3_encode(x), np.array([e4m3_encode_scalar(v) for v in x], np.uint8))
