"""Pins for oracle.select: hand fixture, rank-by-counting brute force, properties."""
import json
import os

import numpy as np
import pytest

from conftest import GOLDEN
from oracle import forced_blocks, select_blocks


def _beats(sa, a, sb, b):
    """True when block a (score sa) ranks ahead of block b (score sb)."""
    na, nb = np.isnan(sa), np.isnan(sb)
    if na or nb:
        return (not na and nb) or (na and nb and a < b)
    return sa > sb or (sa == sb and a < b)


def _brute(scores, nb, budget, n_sink, n_recent):
    if nb <= budget:
        return list(range(nb))
    forced = set(range(min(n_sink, nb))) | set(range(max(0, nb - n_recent), nb))
    rest = [b for b in range(nb) if b not in forced]
    k = budget - len(forced)
    chosen = [b for b in rest if sum(_beats(scores[c], c, scores[b], b) for c in rest if c != b) < k]
    return sorted(forced | set(chosen))


def test_golden():
    with open(os.path.join(GOLDEN, "select_small.json")) as f:
        g = json.load(f)
    scores = np.array([float(x) for x in g["scores"]], np.float32)
    for case in g["cases"]:
        got = select_blocks(scores, len(scores), case["budget"], g["n_sink"], g["n_recent"])
        assert got.tolist() == case["expected"], case["why"]


@pytest.mark.parametrize("seed", range(6))
def test_against_rank_counting(seed):
    rng = np.random.default_rng(seed)
    nb = int(rng.integers(5, 90))
    budget = int(rng.integers(3, 40))
    n_sink, n_recent = int(rng.integers(0, 3)), int(rng.integers(0, 3))
    if n_sink + n_recent > budget:
        n_sink = n_recent = 0
    # coarse values make ties common; sprinkle specials
    scores = rng.integers(-4, 5, size=nb).astype(np.float32)
    specials = np.array([np.nan, np.inf, -np.inf, -0.0, 0.0], np.float32)
    idx = rng.integers(0, nb, size=min(nb, 6))
    scores[idx] = specials[rng.integers(0, len(specials), size=len(idx))]
    got = select_blocks(scores, nb, budget, n_sink, n_recent)
    assert got.tolist() == _brute(scores, nb, budget, n_sink, n_recent)
    assert len(got) == min(budget, nb)
    assert set(forced_blocks(nb, budget, n_sink, n_recent).tolist()) <= set(got.tolist())
    assert np.all(np.diff(got) > 0)


def test_all_equal_scores_take_lowest_indices():
    got = select_blocks(np.zeros(100, np.float32), 100, 10, 1, 2)
    assert got.tolist() == [0, 1, 2, 3, 4, 5, 6, 7, 98, 99]
