"""The workloads' step-to-step selection overlap |S_t & S_t-1| / |S_t| sits where the pages put it
(elastic loading sees more than 80% overlap between steps: tuntang.top survey, section 2.1), and
the budget sweep's calibrated rho values reach their 50 / 80 / 95% targets.  Measured on the
oracle's selections of request 0 (a one-request slice of each workload, as the rho values were
calibrated); the MLA case also keeps its ~50% adjacent-layer overlap."""
import numpy as np
import pytest

import workload as W
from oracle import block_scores, index_keys, select_blocks


def _overlaps(w, steps, layers=1, adjacent=False):
    w = w.with_(n_req=1, n_layer=layers)
    k, _ = W.kv_numpy(w)
    qs = W.QueryStream(w)
    g = w.group
    ik = {(l, h): index_keys(k[l, 0, h], w.ctx0, w.block_size) for l in range(layers) for h in range(w.n_kv_head)}
    nb = ik[(0, 0)].shape[0]
    prev, step_ov, layer_ov = {}, [], []
    for t in range(steps):
        q = qs.queries(t)
        d = qs.drafts(t) if w.lookahead else None
        sels = {}
        for l in range(layers):
            for h in range(w.n_kv_head):
                rows = d[l, 0, :, h * g:(h + 1) * g].reshape(-1, w.d_k) if w.lookahead else q[l, 0, h * g:(h + 1) * g]
                s, _ = block_scores(rows, ik[(l, h)], w.softmax_scale)
                sel = select_blocks(s.astype(np.float32), nb, w.budget_blocks, w.n_sink, w.n_recent)
                if (l, h) in prev:
                    step_ov.append(len(np.intersect1d(prev[(l, h)], sel)) / len(sel))
                prev[(l, h)] = sels[(l, h)] = sel
        if adjacent:
            for l in range(1, layers):
                for h in range(w.n_kv_head):
                    layer_ov.append(len(np.intersect1d(sels[(l - 1, h)], sels[(l, h)])) / len(sels[(l, h)]))
    return float(np.mean(step_ov)), (float(np.mean(layer_ov)) if layer_ov else None)


def test_llama8b_32k_lookahead_overlap():
    ov, _ = _overlaps(W.LLAMA8B_32K, steps=10)
    assert 0.82 <= ov <= 0.92, ov


def test_llama8b_128k_overlap():
    ov, _ = _overlaps(W.LONG_128K, steps=10)
    assert 0.80 <= ov <= 0.90, ov


def test_mla_128k_step_and_adjacent_layer_overlap():
    ov, adj = _overlaps(W.MLA_128K, steps=4, layers=2, adjacent=True)
    assert 0.80 <= ov <= 0.92, ov
    assert 0.45 <= adj <= 0.55, adj


@pytest.mark.parametrize("bs,budget,target", [(16, 2048, 50), (16, 2048, 80), (16, 512, 95), (64, 4096, 80)])
def test_sweep_calibration(bs, budget, target):
    ov, _ = _overlaps(W.get(f"sweep_bs{bs}_b{budget}_ov{target}"), steps=10)
    assert abs(ov - target / 100) <= 0.025, ov


def test_draft_noise_rho_zero_is_independent_noise():
    """draft_rho = 0 reproduces the stateless draft draws exactly; a positive draft_rho keeps the
    noise marginal N(0, sigma^2) but correlates consecutive steps."""
    w = W.TINY_LOOKAHEAD.with_(rho=0.99)
    a, b = W.QueryStream(w), W.QueryStream(w.with_(draft_rho=1e-300))
    for t in range(3):
        assert np.array_equal(a.drafts(t), b.drafts(t))
    c = W.QueryStream(w.with_(draft_rho=0.99))
    d0, d1 = c.drafts(0), c.drafts(1)
    from oracle import bf16_to_f64
    q1, q2 = bf16_to_f64(c.queries(1)), bf16_to_f64(c.queries(2))
    n0 = (bf16_to_f64(d0[:, :, 0]) - q1) / 0.3
    n1 = (bf16_to_f64(d1[:, :, 0]) - q2) / 0.3
    assert 0.8 < n0.std() < 1.2 and 0.8 < n1.std() < 1.2
    assert np.corrcoef(n0.ravel(), n1.ravel())[0, 1] > 0.9
