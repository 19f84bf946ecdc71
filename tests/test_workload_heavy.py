"""The seeded generator's heavy-key sets (input recipe, not the method): independent per-layer sets
by default, chained sets that keep a share of the layer below's positions, and sets shared by all
layers.  These fix the MLA workload's adjacent-layer overlap knob."""
import numpy as np

import workload as W

BASE = W.TINY.with_(name="heavy_sets", n_layer=4, n_kv_head=2, ctx0=4096, n_heavy=200)


def _sets(w, req=0, head=0):
    return [set(W.heavy_positions(w, req, l, head).tolist()) for l in range(w.n_layer)]


def test_sizes_and_range():
    for keep in (0.0, 0.5, 1.0):
        for s in _sets(BASE.with_(heavy_keep=keep)):
            assert len(s) == BASE.n_heavy and min(s) >= 0 and max(s) < BASE.ctx0


def test_keep_zero_reproduces_independent_sets():
    a, b = _sets(BASE), _sets(BASE.with_(heavy_keep=0.0))
    assert a == b
    # independent sets of 200 of 4096 overlap by ~200*200/4096 ~ 10 positions
    assert all(len(a[l] & a[l + 1]) < 40 for l in range(BASE.n_layer - 1))


def test_keep_one_repeats_the_first_layer_and_shared_sets_match_it():
    chained = _sets(BASE.with_(heavy_keep=1.0))
    assert all(s == chained[0] for s in chained)
    shared = _sets(BASE.with_(heavy_shared_layers=True))
    assert all(s == shared[0] for s in shared)
    assert shared[0] == _sets(BASE)[0]          # the shared set is layer 0's shuffle


def test_partial_keep_fraction():
    w = BASE.with_(heavy_keep=0.75, n_heavy=800)
    s = _sets(w)
    for l in range(w.n_layer - 1):
        frac = len(s[l] & s[l + 1]) / w.n_heavy
        # kept share 0.75 (binomial, sd ~0.015) plus the few chance collisions of the refill
        assert 0.70 <= frac <= 0.82, frac


def test_chained_fill_matches_kv_bytes():
    """The heavy rows the K fill scales are the positions heavy_positions reports."""
    import torch
    w = BASE.with_(heavy_keep=0.5, n_layer=2, n_req=1, n_kv_head=1, heavy_scale=64.0)
    k = torch.empty((w.n_layer, 1, 1, w.max_ctx, w.d_k), dtype=torch.int16)
    W.fill_kv(w, k, torch.empty_like(k), 1)
    from oracle import bf16_to_f32
    rows = bf16_to_f32(k.numpy().view(np.uint16))
    for l in range(2):
        norms = np.abs(rows[l, 0, 0, : w.ctx0]).mean(axis=1)
        top = set(np.argsort(-norms)[: w.n_heavy].tolist())
        assert top == set(W.heavy_positions(w, 0, l, 0).tolist())
