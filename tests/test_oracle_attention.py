"""Pins for oracle.attention: torch SDPA (fp64) and closed-form special cases."""
import numpy as np
import torch

from oracle import attend, bf16_to_f32, f32_to_bf16_rne


def _rand(rng, shape, scale=1.0):
    return f32_to_bf16_rne((rng.standard_normal(shape) * scale).astype(np.float32))


def test_matches_sdpa_fp64():
    rng = np.random.default_rng(4)
    q, k, v = _rand(rng, (4, 64)), _rand(rng, (300, 64), 2.0), _rand(rng, (300, 48))
    scale = 0.125
    got = attend(q, k, v, scale)
    tq = torch.from_numpy(bf16_to_f32(q).astype(np.float64))[None, :, None, :]      # (1, G, 1, D)
    tk = torch.from_numpy(bf16_to_f32(k).astype(np.float64))[None, None].expand(1, 4, 300, 64)
    tv = torch.from_numpy(bf16_to_f32(v).astype(np.float64))[None, None].expand(1, 4, 300, 48)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)[0, :, 0].numpy()
    np.testing.assert_allclose(got, ref.astype(np.float32), rtol=0, atol=1e-6)


def test_one_token_returns_v():
    rng = np.random.default_rng(5)
    q, k, v = _rand(rng, (3, 16)), _rand(rng, (1, 16)), _rand(rng, (1, 8))
    np.testing.assert_array_equal(attend(q, k, v, 0.25), np.repeat(bf16_to_f32(v), 3, axis=0))


def test_equal_logits_give_mean_of_v():
    rng = np.random.default_rng(6)
    q = np.zeros((2, 16), np.uint16)                   # q = 0 -> all logits 0
    k, v = _rand(rng, (50, 16)), _rand(rng, (50, 8))
    np.testing.assert_allclose(attend(q, k, v, 1.0), np.repeat(bf16_to_f32(v).astype(np.float64).mean(0, keepdims=True), 2, 0), atol=1e-6)


def test_no_tokens_is_zero():
    out = attend(np.zeros((2, 8), np.uint16), np.zeros((0, 8), np.uint16), np.zeros((0, 4), np.uint16), 1.0)
    assert out.shape == (2, 4) and not out.any()
