"""GPU parity of the fused decode step (kvs_decode_step, with append, prefetch and the
lookahead pipeline) against the oracle, step after step.

Integer-valued inputs make every block score exact in fp32 on both sides, so selections,
cache state and counters must agree bit for bit at every step; attention outputs agree within
2e-3.  With N(0,1) inputs the two sides may order near-tied blocks differently: those units
are checked for a valid selection instead, and compared exactly until their first near-tie."""
import numpy as np
import pytest

import workload as W
from kvs_harness import STAT_KEYS, GpuCase, compare_step as _compare_step

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

INT_CASES = [
    (W.TINY.with_(name="tiny_int", n_req=2, int_scale=2.0), [4096, 3001], False),
    (W.TINY_LOOKAHEAD.with_(name="tiny_la_int", n_req=2, int_scale=2.0), [4096, 3001], False),
    (W.TINY_LOOKAHEAD.with_(name="tiny_la_int_cs", n_req=2, int_scale=2.0), [4096, 2050], True),
    # three layers: each layer's selection chain overlaps the attention of the layers around it
    (W.TINY_LOOKAHEAD.with_(name="tiny_la3_int_cs", n_req=2, n_layer=3, int_scale=2.0), [4096, 1777], True),
    (W.TINY_APPEND.with_(name="tiny_app_int", n_req=2, int_scale=2.0), [4096, 1000], False),
    (W.TINY_PREFETCH.with_(name="tiny_pf_int", n_req=2, int_scale=2.0), [4096, 4095], False),
    (W.TINY_PREFETCH.with_(name="tiny_pf_int_cs", n_req=2, n_layer=3, int_scale=2.0), [4096, 3333], True),
    (W.TINY_MLA.with_(name="tiny_mla_int", n_layer=2, layer_prefetch=True, rho_layer=0.8, int_scale=2.0,
                      steps=12), [4096], False),
    (W.TINY.with_(name="tiny_bs64_int", n_req=2, block_size=64, ctx0=4000, budget_blocks=8, cap_blocks=10,
                  int_scale=2.0), [4000, 3900], False),
    # least-important-first eviction by the step's block scores
    (W.TINY.with_(name="tiny_imp_int", n_req=2, int_scale=2.0, evict_policy="importance"), [4096, 3001], False),
    (W.TINY_LOOKAHEAD.with_(name="tiny_la_imp_int_cs", n_req=2, int_scale=2.0, evict_policy="importance"),
     [4096, 2050], True),
    # [max | min] block summaries scored by the upper bound, with append (the last block's summary
    # is kept up to date) and in lookahead mode
    (W.TINY_APPEND.with_(name="tiny_app_bound_int", n_req=2, int_scale=2.0, score_mode="bound"), [4096, 1000], False),
    (W.TINY_LOOKAHEAD.with_(name="tiny_la_bound_int_cs", n_req=2, int_scale=2.0, score_mode="bound"),
     [4096, 2050], True),
    # E4M3 history and slot pools (integer values up to 16 and power-of-two scales are exact in
    # E4M3, so selections and state stay bit-exact), with append and in lookahead mode
    (W.TINY_APPEND.with_(name="tiny_app_fp8_int", n_req=2, int_scale=2.0, int_clip=4.0, kv_dtype="fp8", k_scale=0.5,
                         v_scale=2.0), [4096, 1000], False),
    (W.TINY_LOOKAHEAD.with_(name="tiny_la_fp8_int_cs", n_req=2, int_scale=2.0, int_clip=4.0, kv_dtype="fp8"),
     [4096, 2050], True),
    # sync steps with a copy stream: the attention over the hits runs while the misses are fetched,
    # then the attention over the fetched blocks merges both parts
    (W.TINY.with_(name="tiny_int_cs", n_req=2, int_scale=2.0), [4096, 3001], True),
    (W.TINY_APPEND.with_(name="tiny_app_int_cs", n_req=2, int_scale=2.0), [4096, 1000], True),
    (W.TINY.with_(name="tiny_bs64_int_cs", n_req=2, block_size=64, ctx0=4000, budget_blocks=8, cap_blocks=10,
                  int_scale=2.0), [4000, 3900], True),
    (W.TINY.with_(name="tiny_imp_int_cs", n_req=2, int_scale=2.0, evict_policy="importance"), [4096, 3001], True),
    (W.TINY_APPEND.with_(name="tiny_app_bound_int_cs", n_req=2, int_scale=2.0, score_mode="bound"), [4096, 1000],
     True),
    (W.TINY_APPEND.with_(name="tiny_app_fp8_int_cs", n_req=2, int_scale=2.0, int_clip=4.0, kv_dtype="fp8",
                         k_scale=0.5, v_scale=2.0), [4096, 1000], True),
    # the sweep's block size 16 / 2048-token budget unit shape (4096 blocks, K_b 128, C 160): the
    # fused top-K + update kernel's dynamic shared memory is just under 48 KB there, and with its
    # static shared memory above it
    (W.sweep_workload(16, 2048, 0.98, n_layer=1, name="sweep16_2048_int").with_(n_req=2, n_q_head=8, n_kv_head=2,
                                                                              steps=6, int_scale=2.0),
     [65536, 60001], True),
]


@pytest.mark.parametrize("w,lens,copy_stream", INT_CASES, ids=[c[0].name for c in INT_CASES])
def test_decode_step_integer_inputs_bit_exact(w, lens, copy_stream):
    g = GpuCase(w, lens, copy_stream=copy_stream)
    o = g.oracle()
    cum = {l: {k: 0 for k in STAT_KEYS} for l in range(w.n_layer)}
    for t in range(min(w.steps, 16)):
        q, d, nk, nv = g.step_inputs(t)
        g.gpu_step(q, d, nk, nv)
        out_ref, recs = o.step(q, d, nk, nv)
        _compare_step(g, o, out_ref, recs, cum, exact=True)
    assert g.ctx.poll_error() == 0


GRAPH_CASES = [
    (W.TINY_LOOKAHEAD.with_(name="tiny_la3_graph", n_req=2, n_layer=3, int_scale=2.0), [4096, 2050]),
    (W.TINY_APPEND.with_(name="tiny_app2_graph", n_req=2, n_layer=2, int_scale=2.0), [4096, 1000]),
]


@pytest.mark.parametrize("w,lens", GRAPH_CASES, ids=[c[0].name for c in GRAPH_CASES])
def test_captured_step_replays_bit_exact(w, lens):
    """The whole step captured once as a CUDA graph over fixed input buffers (as a serving loop
    runs it, with the fetch and the selection chain on their own streams) and replayed step after
    step: selections, cache state, counters and outputs follow the oracle exactly."""
    g = GpuCase(w, lens, copy_stream=True)
    o = g.oracle()
    cum = {l: {k: 0 for k in STAT_KEYS} for l in range(w.n_layer)}
    q, d, nk, nv = g.step_inputs(0)
    g.gpu_step(q, d, nk, nv)
    out_ref, recs = o.step(q, d, nk, nv)
    _compare_step(g, o, out_ref, recs, cum, exact=True)
    B, NL = w.n_req, w.n_layer
    qf = torch.empty((NL, B, w.n_q_head, w.d_k), dtype=torch.int16, device="cuda")
    df = torch.empty((NL, B, w.n_draft, w.n_q_head, w.d_k), dtype=torch.int16, device="cuda") if w.lookahead else None
    kf = torch.empty((NL, B, w.n_kv_head, w.d_k), dtype=torch.int16, device="cuda") if w.append else None
    vf = torch.empty((NL, B, w.n_kv_head, w.d_v), dtype=torch.int16, device="cuda") if w.append else None
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        if w.append:
            g.ctx.advance_ctx(g.ctx_len, stream=s)
        for l in range(NL):
            g.ctx.decode_step(l, qf[l], None if df is None else df[l], w.n_score_q if df is not None else 1, g.index,
                              g.ctx_len, g.out[l], g.stats, None if kf is None else kf[l],
                              None if vf is None else vf[l], g.sel[l], g.nsel[l], stream=s,
                              copy_stream=g.copy_stream)
        g.ctx.join(s)
    for t in range(1, 8):
        q, d, nk, nv = g.step_inputs(t)
        qf.copy_(torch.from_numpy(q.view(np.int16)))
        if df is not None:
            df.copy_(torch.from_numpy(d.view(np.int16)))
        if kf is not None:
            kf.copy_(torch.from_numpy(nk.view(np.int16)))
            vf.copy_(torch.from_numpy(nv.view(np.int16)))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        out_ref, recs = o.step(q, d, nk, nv)
        _compare_step(g, o, out_ref, recs, cum, exact=True)
    assert g.ctx.poll_error() == 0


GAUSS_CASES = [W.TINY.with_(n_req=2), W.TINY_LOOKAHEAD.with_(n_req=2), W.TINY_APPEND, W.TINY_PREFETCH,
               W.TINY_MLA.with_(steps=8), W.TINY_APPEND.with_(name="tiny_append_fp8", kv_dtype="fp8", v_scale=0.5)]


@pytest.mark.parametrize("w", GAUSS_CASES, ids=[c.name for c in GAUSS_CASES])
def test_decode_step_gaussian_inputs(w):
    lens = [w.ctx0] * w.n_req
    g = GpuCase(w, lens)
    o = g.oracle()
    frozen = set()
    for t in range(min(w.steps, 12)):
        q, d, nk, nv = g.step_inputs(t)
        g.gpu_step(q, d, nk, nv)
        out_ref, recs = o.step(q, d, nk, nv)
        _compare_step(g, o, out_ref, recs, None, exact=False, frozen=frozen)
    # near-ties are rare: most units must have stayed in lock-step
    n_units = w.n_layer * w.n_req * w.n_kv_head
    assert len(frozen) <= max(1, n_units // 2)
    assert g.ctx.poll_error() == 0


def test_rebind_after_recollapse_keeps_parity():
    """The host history can be re-registered and bound again between steps (what a caller does
    after remapping split huge pages): the cache state stays valid and steps stay bit-exact."""
    import sparse_kv_cache_decode_gb300 as K
    # 1 GiB of history, so it lives in a huge-page HostArray; 32768 blocks per unit: two-phase top-K
    w = W.TINY.with_(name="tiny_rebind", n_req=2, ctx0=524288, steps=6, int_scale=2.0)
    g = GpuCase(w, [524288, 400001])
    assert g._arrays, "expected a huge-page host array"
    o = g.oracle()
    cum = {l: {k: 0 for k in STAT_KEYS} for l in range(w.n_layer)}
    for t in range(w.steps):
        if t == 3:
            for a in g._arrays:
                assert isinstance(a, K.HostArray)
                a.recollapse()
            g.ctx.bind_host_kv(g.k_host, g.v_host)
        q, d, nk, nv = g.step_inputs(t)
        g.gpu_step(q, d, nk, nv)
        out_ref, recs = o.step(q, d, nk, nv)
        _compare_step(g, o, out_ref, recs, cum, exact=True)
    assert g.ctx.poll_error() == 0
    g.close()
