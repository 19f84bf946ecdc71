"""Pins for oracle.index_keys: hand-derived fixture, bs = 1 identity, exact means."""
import json
import os

import numpy as np

from conftest import GOLDEN
from oracle import bf16_to_f32, f32_to_bf16_rne, index_keys


def _load():
    with open(os.path.join(GOLDEN, "index_keys_small.json")) as f:
        return json.load(f)


def test_golden_cases():
    for case in _load()["cases"]:
        keys = f32_to_bf16_rne(np.array(case["keys"], np.float32))
        assert np.array_equal(bf16_to_f32(keys), np.array(case["keys"], np.float32)), "fixture keys must be bf16-exact"
        ik = index_keys(keys, case["ctx_len"], case["block_size"])
        if "expected" in case:
            np.testing.assert_array_equal(bf16_to_f32(ik), np.array(case["expected"], np.float32), err_msg=case["name"])
        else:
            np.testing.assert_array_equal(ik, np.array(case["expected_bits"], np.uint16), err_msg=case["name"])


def test_block_size_one_is_identity():
    rng = np.random.default_rng(1)
    k = f32_to_bf16_rne(rng.standard_normal((37, 24)).astype(np.float32))
    np.testing.assert_array_equal(index_keys(k, 37, 1), k)


def test_exact_means_of_small_integers():
    # integers below 2^8 are bf16-exact and sums of 16 of them are exact in fp32: the mean
    # equals the exact rational mean rounded once to bf16.
    rng = np.random.default_rng(2)
    vals = rng.integers(-100, 100, size=(53, 8)).astype(np.float32)
    k = f32_to_bf16_rne(vals)
    ik = index_keys(k, 53, 16)
    for b in range(4):
        rows = vals[b * 16: min(53, (b + 1) * 16)]
        exact = rows.astype(np.float64).sum(0) / rows.shape[0]
        np.testing.assert_array_equal(ik[b], f32_to_bf16_rne(exact.astype(np.float32)))


def test_partial_block_uses_present_count():
    k = f32_to_bf16_rne(np.array([[3.0], [3.0], [6.0]], np.float32))
    ik = index_keys(k, 3, 4)
    assert bf16_to_f32(ik)[0, 0] == 4.0   # (3 + 3 + 6) / 3, not / 4
