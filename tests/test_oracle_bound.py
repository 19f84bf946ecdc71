"""Pins for oracle.bound: the hand-worked fixture, the upper-bound property against brute force
over every token, equality on one-token blocks, and [k | k] summaries of one-token blocks."""
import json
import os

import numpy as np

from conftest import GOLDEN
from oracle import (bf16_to_f64, block_scores, block_scores_bound, f32_to_bf16_rne, index_keys, index_minmax,
                    index_minmax_block)


def _bf(x):
    return f32_to_bf16_rne(np.asarray(x, np.float32))


def test_hand_worked_fixture():
    with open(os.path.join(GOLDEN, "bound_small.json")) as f:
        g = json.load(f)
    k = _bf(g["keys"])
    summ = index_minmax(k, g["ctx_len"], g["block_size"])
    np.testing.assert_array_equal(bf16_to_f64(summ), np.array(g["summaries"]))
    s, a = block_scores_bound(_bf(g["rows"]), summ, g["scale"])
    np.testing.assert_array_equal(s, g["scores"])
    np.testing.assert_array_equal(a, g["bounds_A"])


def test_bound_is_an_upper_bound_of_every_token_logit():
    rng = np.random.default_rng(11)
    for trial in range(30):
        d, bs = int(rng.choice([4, 8, 16])), int(rng.integers(1, 9))
        L = int(rng.integers(1, 60))
        k = _bf(rng.normal(size=(L, d)) * rng.choice([0.5, 3.0]))
        q = _bf(rng.normal(size=(int(rng.integers(1, 5)), d)))
        summ = index_minmax(k, L, bs)
        s, _ = block_scores_bound(q, summ, 1.0)
        logits = bf16_to_f64(q) @ bf16_to_f64(k).T                  # (R, L)
        nb = (L + bs - 1) // bs
        for b in range(nb):
            tok_max = logits[:, b * bs: min(L, (b + 1) * bs)].max()
            assert s[b] >= tok_max - 1e-12 * (1 + abs(tok_max))
            if min(L, (b + 1) * bs) - b * bs == 1:                  # one token: the bound is exact
                assert s[b] == tok_max


def test_one_token_blocks_summarise_to_the_key_and_match_mean_scoring():
    rng = np.random.default_rng(5)
    k = _bf(rng.normal(size=(9, 8)))
    q = _bf(rng.normal(size=(3, 8)))
    summ = index_minmax(k, 9, 1)
    np.testing.assert_array_equal(summ, np.concatenate([k, k], axis=1))
    s_b, _ = block_scores_bound(q, summ, 0.25)
    s_m, _ = block_scores(q, index_keys(k, 9, 1), 0.25)
    np.testing.assert_array_equal(s_b, s_m)


def test_ragged_last_block_uses_present_rows_only():
    k = _bf([[1.0, 1.0], [2.0, -3.0], [9.0, 9.0]])
    np.testing.assert_array_equal(bf16_to_f64(index_minmax_block(k[:2])), [2.0, 1.0, 1.0, -3.0])
    summ = index_minmax(k, 2, 2)                                     # the third row is past the end
    assert summ.shape == (1, 4)
    np.testing.assert_array_equal(bf16_to_f64(summ[0]), [2.0, 1.0, 1.0, -3.0])
