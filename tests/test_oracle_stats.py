"""Pin of the decode-step oracle's per-layer counters (OracleDecoder.stats) against hand-worked
cases (tests/golden/stats_small.json): a ragged last block whose fetch counts only its present
rows, a cross-layer prefetch that evicts and is then hit, and a lookahead bootstrap step whose
two updates both count, followed by a pin fallback.  The keys are one-hot per block, so each
query fixes the selection exactly and every counter follows by hand from the cache rules."""
import json
import os

import numpy as np

import workload as W
from oracle import OracleDecoder, f32_to_bf16_rne

from conftest import GOLDEN

with open(os.path.join(GOLDEN, "stats_small.json")) as f:
    G = json.load(f)

SH = G["shape"]
ONE = int(f32_to_bf16_rne(np.array([1.0], np.float32))[0])


def _workload(case):
    return W.Workload(name="stats_pin", n_req=1, n_layer=case["n_layer"], n_q_head=SH["n_q_head"],
                      n_kv_head=SH["n_kv_head"], d_k=SH["d_k"], d_v=SH["d_v"], block_size=SH["block_size"],
                      ctx0=SH["ctx0"], steps=len(case["steps"]), budget_blocks=SH["budget_blocks"],
                      n_sink=SH["n_sink"], n_recent=SH["n_recent"], cap_blocks=SH["cap_blocks"],
                      lookahead=case["lookahead"], n_draft=case.get("n_draft", 0),
                      layer_prefetch=case["layer_prefetch"])


def _history(w):
    """Block b < 7 holds key e_b in every token; the ragged block 7 holds zero keys; V = 1."""
    k = np.zeros((w.n_layer, 1, 1, w.max_ctx, w.d_k), np.uint16)
    for t in range(w.ctx0):
        b = t // w.block_size
        if b < 7:
            k[:, 0, 0, t, b] = ONE
    v = np.full((w.n_layer, 1, 1, w.max_ctx, w.d_v), ONE, np.uint16)
    return k, v


def _rows(spec, d):
    q = np.zeros(d, np.float32)
    for b, val in spec.items():
        q[int(b)] = val
    return f32_to_bf16_rne(q)


def _run(case):
    w = _workload(case)
    assert w.max_ctx == SH["ctx0"] and w.max_blocks == 8
    k, v = _history(w)
    dec = OracleDecoder(w, k, v, [w.ctx0])
    assert dec.row_bytes() == SH["row_bytes"]
    for step in case["steps"]:
        q = np.zeros((w.n_layer, 1, 1, w.d_k), np.uint16)
        for l, spec in step["query_top"].items():
            q[int(l), 0, 0] = _rows(spec, w.d_k)
        drafts = None
        if w.lookahead:
            drafts = np.zeros((w.n_layer, 1, 1, 1, w.d_k), np.uint16)
            for l, spec in step["draft_top"].items():
                drafts[int(l), 0, 0, 0] = _rows(spec, w.d_k)
        _, recs = dec.step(q, drafts)
        yield step, recs, dec.stats()


def test_stats_sync_prefetch_ragged():
    case = G["cases"][0]
    for step, recs, st in _run(case):
        for l, sel in step["sel"].items():
            assert recs[(int(l), 0, 0)].sel.tolist() == sel
        for l, want in step["stats"].items():
            assert st[int(l)] == want, (step["derivation"], st[int(l)], want)


def test_stats_lookahead_bootstrap_and_pin_fallback():
    case = G["cases"][1]
    for step, recs, st in _run(case):
        rec = recs[(0, 0, 0)]
        assert rec.attn_sel.tolist() == step["attn_sel"]["0"]
        assert rec.sel.tolist() == step["sel"]["0"]
        assert st[0] == step["stats"]["0"], (step["derivation"], st[0])


def test_bytes_fetched_counts_present_rows_only():
    """The ragged block's fetch is 2 rows, not a full block: a planted full-block count (the mistake
    of charging bs rows for every block) would give 384 bytes for the first step of layer 0."""
    case = G["cases"][0]
    step, recs, st = next(_run(case))
    assert st[0]["bytes_fetched"] == 2 * SH["bytes_full_block"] + SH["bytes_block_7"]
