"""Pins for oracle.scores: exactly rounded sums, the single-row reduction, the group max."""
import math

import numpy as np

from oracle import bf16_to_f64, block_scores, f32_to_bf16_rne


def _rand_bf16(rng, shape, scale=1.0):
    return f32_to_bf16_rne((rng.standard_normal(shape) * scale).astype(np.float32))


def test_against_fsum_bruteforce():
    rng = np.random.default_rng(3)
    q = _rand_bf16(rng, (6, 40))
    ik = _rand_bf16(rng, (25, 40))
    scale = 0.125
    s, a = block_scores(q, ik, scale)
    qf, kf = bf16_to_f64(q), bf16_to_f64(ik)
    for b in range(25):
        dots = [math.fsum(qf[r, d] * kf[b, d] for d in range(40)) for r in range(6)]
        absd = [math.fsum(abs(qf[r, d] * kf[b, d]) for d in range(40)) for r in range(6)]
        assert abs(s[b] - scale * max(dots)) <= 1e-12 * (1 + scale * max(absd))
        assert abs(a[b] - scale * max(absd)) <= 1e-12 * (1 + scale * max(absd))


def test_single_row_is_scaled_dot_product():
    q = f32_to_bf16_rne(np.array([[2.0, 0.0, 0.0, 0.0]], np.float32))
    ik = f32_to_bf16_rne(np.array([[3.0, 1.0, 0.0, 0.0], [-1.0, 5.0, 0.0, 0.0]], np.float32))
    s, a = block_scores(q, ik, 1.0 / math.sqrt(4))
    np.testing.assert_allclose(s, [3.0, -1.0])
    np.testing.assert_allclose(a, [3.0, 1.0])


def test_group_max_not_mean_or_sum():
    # three rows (e.g. a GQA group x drafts); block 0 favoured by row 2 only
    q = f32_to_bf16_rne(np.array([[1, 0], [0, 1], [-4, 0]], np.float32))
    ik = f32_to_bf16_rne(np.array([[-1, 0], [1, 1]], np.float32))
    s, _ = block_scores(q, ik, 1.0)
    np.testing.assert_allclose(s, [4.0, 1.0])     # max over rows: 4 (row 2) and 1
