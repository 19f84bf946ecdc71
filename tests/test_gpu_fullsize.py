"""GPU parity at the workloads' full sizes, in the launch configuration bench.py times.

Each test binds the whole host history and runs the fused step for a few steps (lookahead with
the fetch on a side stream for the 8B case, append with the fetch on a side stream beside the
attention over the hits for the 128K case, prefetch for the MLA case).
The oracle recomputes one sampled request in full (every layer and kv head) step by step; for
every unit the size-independent properties are checked: selection count, order, range and forced
blocks, and the bytes of resident slots against the host history."""
import numpy as np
import pytest

import workload as W
from kvs_harness import GpuCase, compare_step
from oracle import forced_blocks

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")


def _properties(g, step_seed):
    w = g.w
    sel = g.sel.cpu().numpy()
    nsel = g.nsel.cpu().numpy()
    lens = g.ctx_len.cpu().numpy()
    for l in range(w.n_layer):
        for r in range(w.n_req):
            nb = (int(lens[r]) + w.block_size - 1) // w.block_size
            forced = set(forced_blocks(nb, w.budget_blocks, w.n_sink, w.n_recent).tolist())
            for h in range(w.n_kv_head):
                n = int(nsel[l, r, h])
                s = sel[l, r, h, :n]
                assert n == min(w.budget_blocks, nb)
                assert np.all(np.diff(s) > 0) and s[0] >= 0 and s[-1] < nb
                assert forced <= set(s.tolist())
    # resident slot bytes equal the host rows, for a few random units of a random layer
    rng = np.random.default_rng(step_seed)
    l = int(rng.integers(0, w.n_layer))
    b2s, _, _, _ = g.ctx.cache_export(l)
    kp, vp = g.ctx.slot_pool_tensors(l)
    for u in rng.choice(g.ctx.units, min(4, g.ctx.units), replace=False):
        r, h = divmod(int(u), w.n_kv_head)
        L = int(lens[r])
        blocks = np.nonzero(b2s[u] >= 0)[0]
        for b in rng.choice(blocks, min(6, len(blocks)), replace=False):
            s = int(b2s[u, b])
            rows = min(w.block_size, L - int(b) * w.block_size)
            t0 = int(b) * w.block_size
            np.testing.assert_array_equal(kp[u, s, :rows].cpu().numpy().view(np.uint16), g.k_np[l, r, h, t0:t0 + rows])
            if vp is not None:
                np.testing.assert_array_equal(vp[u, s, :rows].cpu().numpy().view(np.uint16),
                                              g.v_np[l, r, h, t0:t0 + rows])


def _run(w, steps, copy_stream=False, reqs=(0,)):
    g = GpuCase(w, copy_stream=copy_stream)
    try:
        o = g.oracle(list(reqs))
        frozen = set()
        for t in range(steps):
            q, d, nk, nv = g.step_inputs(t)
            g.gpu_step(q, d, nk, nv)
            out_ref, recs = o.step(q, d, nk, nv)
            compare_step(g, o, out_ref, recs, None, exact=False, frozen=frozen)
            _properties(g, 1000 + t)
        n_units = w.n_layer * len(reqs) * w.n_kv_head
        assert len(frozen) <= n_units // 4, f"{len(frozen)} of {n_units} sampled units hit near-ties"
        assert g.ctx.poll_error() == 0
    finally:
        g.close()


def test_llama8b_32k_lookahead_full():
    _run(W.LLAMA8B_32K, steps=4, copy_stream=True)


def test_llama8b_128k_append_full():
    _run(W.LONG_128K.with_(steps=8), steps=3, copy_stream=True)


def test_mla_128k_token_topk_full():
    _run(W.MLA_128K.with_(steps=4), steps=2)


def test_sweep_bs16_budget2048_full():
    _run(W.sweep_workload(16, 2048, 0.9), steps=2)


def test_sweep_bs64_budget2048_full():
    # block 64: four 16-row sub-tiles per block in the attention kernel
    _run(W.sweep_workload(64, 2048, 0.9, n_layer=4), steps=2)


def test_sweep_bs16_budget4096_full():
    # K_b 256, cache 320 slots: the largest budget of the sweep
    _run(W.sweep_workload(16, 4096, 0.9, n_layer=4), steps=2)
