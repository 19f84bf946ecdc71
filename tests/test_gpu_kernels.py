"""GPU parity of each libkvs entry point against the CPU oracle (run on a GB300).

Each stage is fed inputs that come from the seeded generator or from the oracle, never from
another GPU stage, and compared with the oracle stage: bit-exact for index keys, selections
and cache state; within 1e-4 (|s| + A) for scores; within 2e-3 absolute for attention."""
import math

import numpy as np
import pytest

import workload as W
from kvs_harness import GpuCase, score_tolerance
from oracle import (UnitCache, attend, bf16_to_f32, block_scores, block_scores_bound, cache_update, index_keys,
                    index_minmax, layer_prefetch, select_blocks)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

MLA_G128 = W.MLA_128K.with_(name="mla_g128_small", n_req=2, n_layer=1, ctx0=2048, steps=4, budget_blocks=256,
                            cap_blocks=384, n_heavy=20)
# 64 heads per latent row: the mma.sync MLA kernel; 128 heads: the tcgen05 kernel, here with 8 units
# so that each CTA runs 8 tiles of 32 tokens (the stage ring wraps; ragged last tile)
MLA_G64 = MLA_G128.with_(name="mla_g64_small", n_q_head=64)
MLA_G128_B8 = MLA_G128.with_(name="mla_g128_b8", n_req=8, ctx0=4096, budget_blocks=2048, cap_blocks=2304, n_heavy=40)
TINY3 = W.TINY.with_(name="tiny3", n_req=3)
TINY_G8 = W.TINY.with_(name="tiny_g8", n_req=2, n_q_head=16, n_kv_head=2)
TINY_BS64 = W.TINY.with_(name="tiny_bs64", n_req=2, block_size=64, ctx0=3000, budget_blocks=8, cap_blocks=12)
# 16 query heads per kv head x 5 scoring queries: 80 rows per unit (the tensor-memory scoring path)
TINY_LA_G16 = W.TINY_LOOKAHEAD.with_(name="tiny_la_g16", n_req=3, n_q_head=32, n_kv_head=2)
# [max | min] summaries with the upper-bound score: 8B-like rows on the mma.sync path, 80 rows per
# unit on the tensor-memory path
TINY3_BOUND = TINY3.with_(name="tiny3_bound", score_mode="bound")
TINY_LA_G16_BOUND = TINY_LA_G16.with_(name="tiny_la_g16_bound", score_mode="bound")


def _summaries(w, k_rows, L):
    return index_minmax(k_rows, L, w.block_size) if w.score_mode == "bound" else index_keys(k_rows, L, w.block_size)


def _scores(w, rows, summ):
    return (block_scores_bound if w.score_mode == "bound" else block_scores)(rows, summ, w.softmax_scale)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def _nb(L, bs):
    return (L + bs - 1) // bs


TINY3_FP8 = TINY3.with_(name="tiny3_fp8", kv_dtype="fp8", k_scale=0.5, v_scale=0.25)


@pytest.mark.parametrize("w,lens", [(TINY3, [4096, 1000, 17]), (W.TINY_MLA, [4096]),
                                    (TINY_BS64, [3000, 2999]), (MLA_G128, [2048, 333]), (TINY3_FP8, [4096, 1000, 17]),
                                    (TINY3_BOUND, [4096, 1000, 17]), (TINY_BS64.with_(score_mode="bound"), [3000, 7])])
def test_index_build_bit_exact(w, lens):
    g = GpuCase(w, lens)
    idx = g.index.cpu().numpy().view(np.uint16)
    for l in range(w.n_layer):
        for r, L in enumerate(lens):
            for h in range(w.n_kv_head):
                nb = _nb(L, w.block_size)
                if w.kv_dtype == "fp8":
                    from oracle.fp8 import dequantize_f32
                    ref = index_keys(dequantize_f32(g.k_np[l, r, h], w.k_scale), L, w.block_size)
                else:
                    ref = _summaries(w, g.k_np[l, r, h], L)
                np.testing.assert_array_equal(idx[l, r, h, :nb], ref, err_msg=f"unit {(l, r, h)}")


def _score_rows(w, q, d, l, r, h):
    heads = slice(h * w.group, (h + 1) * w.group)
    if d is None:
        return q[l, r, heads]
    return d[l, r, :, heads].reshape(-1, w.d_k)


@pytest.mark.parametrize("w,lens", [(TINY3, [4096, 1000, 17]), (W.TINY_LOOKAHEAD.with_(n_req=2), [4096, 2222]),
                                    (TINY_G8, [4096, 4000]), (W.TINY_MLA, [4096]), (MLA_G128, [2048, 1500]),
                                    (TINY3.with_(int_scale=2.0), [4096, 1000, 17]),
                                    (TINY_LA_G16, [4096, 1000, 17]),
                                    (TINY_LA_G16.with_(int_scale=2.0), [4096, 2049, 129]),
                                    (MLA_G128.with_(int_scale=1.0), [2048, 1500]),
                                    (TINY3_BOUND, [4096, 1000, 17]), (TINY3_BOUND.with_(int_scale=2.0), [4096, 1000, 17]),
                                    (TINY_LA_G16_BOUND, [4096, 1000, 17]),
                                    (TINY_LA_G16_BOUND.with_(int_scale=2.0), [4096, 2049, 129])])
def test_score_blocks(w, lens):
    g = GpuCase(w, lens)
    scores = torch.full((w.n_req, w.n_kv_head, g.nb_max), float("nan"), dtype=torch.float32, device="cuda")
    for t in range(2):
        q, d, _, _ = g.step_inputs(t)
        src = d if d is not None else q
        nq = w.n_score_q
        for l in range(w.n_layer):
            g.ctx.score_blocks(l, _dev(src[l]), nq, g.index, g.ctx_len, scores)
            got = scores.cpu().numpy()
            for r, L in enumerate(lens):
                for h in range(w.n_kv_head):
                    nb = _nb(L, w.block_size)
                    ik = _summaries(w, g.k_np[l, r, h], L)
                    s, a = _scores(w, _score_rows(w, q, d, l, r, h), ik)
                    gs = got[r, h, :nb].astype(np.float64)
                    if w.int_scale > 0:     # exact integer-valued dot products: bit-exact fp32
                        np.testing.assert_array_equal(got[r, h, :nb], s.astype(np.float32))
                    else:
                        err = np.abs(gs - s)
                        tol = score_tolerance(s, a)
                        assert np.all(err <= tol), f"unit {(l, r, h)} max err/tol {np.max(err / tol)}"


def _special_scores(seed, n):
    u = W.uniform_f32(seed, 7, n, -4.0, 4.0)
    s = np.round(u * 4.0).astype(np.float32) / 4.0          # coarse values: many ties
    pos = W.randint(seed, 8, 12, n)
    specials = np.array([np.nan, np.inf, -np.inf, -0.0, 0.0, np.nan], np.float32)
    for i, p in enumerate(pos):
        s[p] = specials[i % len(specials)]
    return s


@pytest.mark.parametrize("lens,budget,sink,recent,bs", [
    ([4096, 1000, 17], 16, 1, 2, 16),        # ragged, one context below the budget
    ([4096, 4096], 2, 1, 1, 16),              # budget == forced set
    ([300000, 123457], 128, 1, 2, 16),        # > 16384 blocks: two phases over 2 chunks
    ([65536, 65536], 256, 0, 0, 16),          # pure top-k
    ([131072, 70001, 1500], 2048, 0, 0, 1),   # token blocks: 8 chunks, ragged, one below the budget
    ([200000, 16385], 512, 4, 8, 1),          # 13 chunks framed by sink and recent blocks
    ([131072], 4096, 1, 1, 1),                # candidates too many to merge: one pass from global memory
])
def test_topk_select_bit_exact(lens, budget, sink, recent, bs):
    w = W.TINY.with_(name="topk", n_req=len(lens), ctx0=max(lens), budget_blocks=budget, n_sink=sink,
                     n_recent=recent, cap_blocks=budget, n_heavy=0, n_layer=1, block_size=bs)
    g = GpuCase(w, lens)
    nbm = g.nb_max
    host = np.stack([np.stack([_special_scores(17 + r * 7 + h, nbm) for h in range(w.n_kv_head)])
                     for r in range(w.n_req)])
    scores = torch.from_numpy(host).cuda()
    sel = torch.full((w.n_req, w.n_kv_head, budget), -7, dtype=torch.int32, device="cuda")
    nsel = torch.zeros((w.n_req, w.n_kv_head), dtype=torch.int32, device="cuda")
    g.ctx.topk_select(scores, g.ctx_len, sel, nsel)
    gs, gn = sel.cpu().numpy(), nsel.cpu().numpy()
    for r, L in enumerate(lens):
        for h in range(w.n_kv_head):
            nb = _nb(L, w.block_size)
            ref = select_blocks(host[r, h], nb, budget, sink, recent)
            assert gn[r, h] == len(ref)
            np.testing.assert_array_equal(gs[r, h, :len(ref)], ref, err_msg=f"unit {(r, h)}")
    assert g.ctx.poll_error() == 0


def _threshold_dup_scores(seed, n, k, mode):
    """Scores whose k-th largest value (the top-K threshold) recurs a few times: fine values
    ('fine': the threshold's 8-bit digit bin holds a few keys after the second radix pass) or
    values spread over many exponents and both signs ('spread': already after the first)."""
    u = W.uniform_f32(seed, 9, n, 0.0, 1.0).astype(np.float64)
    if mode == "fine":
        s = (0.5 + 2.5 * u).astype(np.float32)
    else:
        e = W.uniform_f32(seed, 10, n, -60.0, 60.0).astype(np.float64)
        sign = np.where(W.uniform_f32(seed, 11, n, 0.0, 1.0) < 0.3, -1.0, 1.0)
        s = (sign * np.exp2(e) * (1.0 + u)).astype(np.float32)
    t = np.sort(s)[::-1][k - 1]
    pos = W.randint(seed, 12, 5, n)
    s[pos] = t                                   # duplicates of the threshold value
    return s


def test_topk_two_phase_guess_falls_back_bit_exact():
    """Two-phase top-K whose unit-wide threshold guess is too high: the scores at the guess's
    evenly spaced sample positions are large and every other score is small, so fewer than k kept
    keys reach the guess and the merge selects again from the scores in global memory."""
    lens, budget = [131072, 131072 - 77], 2048
    w = W.TINY.with_(name="topk_fallback", n_req=len(lens), ctx0=max(lens), budget_blocks=budget, n_sink=0,
                     n_recent=0, cap_blocks=budget, n_heavy=0, n_layer=1, block_size=1)
    g = GpuCase(w, lens)
    nbm = g.nb_max
    host = np.zeros((w.n_req, w.n_kv_head, nbm), np.float32)
    for r, L in enumerate(lens):
        for h in range(w.n_kv_head):
            s = W.uniform_f32(41 + r * 7 + h, 13, nbm, -1.0, 0.0)
            # the guess samples position i * L / 4096 of the unit's L candidates
            samp = (np.arange(4096, dtype=np.int64) * L) // 4096
            s[samp] = 10.0 + W.uniform_f32(42 + r * 7 + h, 14, 4096, 0.0, 1.0)
            host[r, h] = s
    scores = torch.from_numpy(host).cuda()
    sel = torch.full((w.n_req, w.n_kv_head, budget), -7, dtype=torch.int32, device="cuda")
    nsel = torch.zeros((w.n_req, w.n_kv_head), dtype=torch.int32, device="cuda")
    g.ctx.topk_select(scores, g.ctx_len, sel, nsel)
    gs, gn = sel.cpu().numpy(), nsel.cpu().numpy()
    for r, L in enumerate(lens):
        for h in range(w.n_kv_head):
            ref = select_blocks(host[r, h], _nb(L, 1), budget, 0, 0)
            assert gn[r, h] == len(ref)
            np.testing.assert_array_equal(gs[r, h, :len(ref)], ref, err_msg=f"unit {(r, h)}")
    assert g.ctx.poll_error() == 0


@pytest.mark.parametrize("mode", ["fine", "spread"])
def test_topk_select_threshold_ties_bit_exact(mode):
    lens, budget, sink, recent = [32768, 20000, 7001], 128, 1, 2
    w = W.TINY.with_(name="topk_ties", n_req=len(lens), ctx0=max(lens), budget_blocks=budget, n_sink=sink,
                     n_recent=recent, cap_blocks=budget, n_heavy=0, n_layer=1)
    g = GpuCase(w, lens)
    nbm = g.nb_max
    k = budget - sink - recent
    host = np.stack([np.stack([_threshold_dup_scores(31 + r * 5 + h, nbm, k, mode) for h in range(w.n_kv_head)])
                     for r in range(w.n_req)])
    scores = torch.from_numpy(host).cuda()
    sel = torch.full((w.n_req, w.n_kv_head, budget), -7, dtype=torch.int32, device="cuda")
    nsel = torch.zeros((w.n_req, w.n_kv_head), dtype=torch.int32, device="cuda")
    g.ctx.topk_select(scores, g.ctx_len, sel, nsel)
    gs, gn = sel.cpu().numpy(), nsel.cpu().numpy()
    for r, L in enumerate(lens):
        for h in range(w.n_kv_head):
            nb = _nb(L, w.block_size)
            ref = select_blocks(host[r, h], nb, budget, sink, recent)
            assert gn[r, h] == len(ref)
            np.testing.assert_array_equal(gs[r, h, :len(ref)], ref, err_msg=f"unit {(r, h)}")
    assert g.ctx.poll_error() == 0


def _correlated_selections(seed, nb, budget, steps, keep=0.7):
    rng = np.random.default_rng(seed)
    cur = np.sort(rng.choice(nb, min(budget, nb), replace=False))
    out = []
    for _ in range(steps):
        k = cur[rng.random(len(cur)) < keep]
        n_new = min(budget, nb) - len(k)
        fresh = rng.choice(np.setdiff1d(np.arange(nb), k), n_new, replace=False)
        cur = np.sort(np.concatenate([k, fresh]))
        n = len(cur) if rng.random() > 0.15 else max(1, len(cur) - int(rng.integers(0, 3)))
        out.append(cur[:n] if n == len(cur) else np.sort(rng.choice(cur, n, replace=False)))
    return out


def _check_state(g, layer, caches, lens):
    w = g.w
    b2s, s2b, st, clk = g.ctx.cache_export(layer)
    for u in range(g.ctx.units):
        c = caches[u]
        np.testing.assert_array_equal(s2b[u], c.slot2block, err_msg=f"slot2block unit {u}")
        np.testing.assert_array_equal(st[u].astype(np.int64), c.stamp, err_msg=f"stamp unit {u}")
        assert int(clk[u]) == c.clock
        np.testing.assert_array_equal(b2s[u, : c.n_blocks], c.block2slot[: g.nb_max], err_msg=f"block2slot unit {u}")


def _check_slots(g, layer, caches, lens, blocks_by_unit):
    w = g.w
    kp, vp = g.ctx.slot_pool_tensors(layer)
    kp = kp.cpu().numpy().view(g.k_np.dtype)
    vp = None if vp is None else vp.cpu().numpy().view(g.k_np.dtype)
    for u, blocks in blocks_by_unit.items():
        r, h = divmod(u, w.n_kv_head)
        L = lens[r]
        for b in blocks:
            s = caches[u].block2slot[b]
            rows = min(w.block_size, L - b * w.block_size)
            t0 = b * w.block_size
            np.testing.assert_array_equal(kp[u, s, :rows], g.k_np[layer, r, h, t0:t0 + rows], err_msg=f"K slot {u}/{b}")
            if vp is not None:
                np.testing.assert_array_equal(vp[u, s, :rows], g.v_np[layer, r, h, t0:t0 + rows])


@pytest.mark.parametrize("lookahead,cap", [(False, 11), (False, 8), (True, 12), (True, 9)])
def test_cache_update_sequences_bit_exact(lookahead, cap):
    lens = [1000, 997]
    w = W.TINY.with_(name="cache", n_req=2, ctx0=1000, budget_blocks=8, cap_blocks=cap, lookahead=lookahead,
                     n_draft=4 if lookahead else 0)
    g = GpuCase(w, lens)
    U = g.ctx.units
    caches = [UnitCache(cap, g.nb_max) for _ in range(U)]
    seqs = [_correlated_selections(40 + u, _nb(lens[u // w.n_kv_head], 16), 8, 30) for u in range(U)]
    prev = [None] * U
    sel = torch.zeros((w.n_req, w.n_kv_head, 8), dtype=torch.int32, device="cuda")
    nsel = torch.zeros((w.n_req, w.n_kv_head), dtype=torch.int32, device="cuda")
    sos = torch.full((w.n_req, w.n_kv_head, 8), -1, dtype=torch.int32, device="cuda")
    stats = torch.zeros((1, 7), dtype=torch.int64, device="cuda")
    tot = dict(hits=0, misses=0, evictions=0, pin_fallbacks=0)
    for step in range(30):
        hs = np.zeros((U, 8), np.int32)
        hn = np.zeros(U, np.int32)
        for u in range(U):
            s = seqs[u][step]
            hs[u, :len(s)] = s
            hn[u] = len(s)
        sel.copy_(torch.from_numpy(hs.reshape(w.n_req, w.n_kv_head, 8)))
        nsel.copy_(torch.from_numpy(hn.reshape(w.n_req, w.n_kv_head)))
        g.ctx.cache_update(0, sel, nsel, g.ctx_len, sos, stats)
        got_sos = sos.cpu().numpy().reshape(U, 8)
        for u in range(U):
            s = seqs[u][step]
            res = cache_update(caches[u], s, prev[u] if lookahead else None)
            prev[u] = s
            np.testing.assert_array_equal(got_sos[u, :len(s)], res.slot_of_sel, err_msg=f"step {step} unit {u}")
            tot["hits"] += len(res.hits)
            tot["misses"] += len(res.misses)
            tot["evictions"] += res.n_evictions
            tot["pin_fallbacks"] += int(res.pin_fallback)
        _check_state(g, 0, caches, lens)
        _check_slots(g, 0, caches, lens, {u: seqs[u][step] for u in range(U)})
    st = stats.cpu().numpy()[0]
    assert [st[0], st[1], st[2], st[5]] == [tot["hits"], tot["misses"], tot["evictions"], tot["pin_fallbacks"]]
    assert g.ctx.poll_error() == 0


def test_layer_prefetch_sequences_bit_exact():
    lens = [1000, 1000]
    w = W.TINY.with_(name="prefetch", n_req=2, n_layer=2, ctx0=1000, budget_blocks=8, cap_blocks=12,
                     layer_prefetch=True)
    g = GpuCase(w, lens)
    U = g.ctx.units
    caches = [UnitCache(12, g.nb_max) for _ in range(U)]
    sels = [_correlated_selections(70 + u, 63, 8, 25) for u in range(U)]
    hints = [_correlated_selections(90 + u, 63, 8, 25, keep=0.5) for u in range(U)]

    def dev_sel(lists):
        a = np.zeros((U, 8), np.int32)
        n = np.zeros(U, np.int32)
        for u, s in enumerate(lists):
            a[u, :len(s)] = s
            n[u] = len(s)
        return (torch.from_numpy(a.reshape(w.n_req, w.n_kv_head, 8)).cuda(),
                torch.from_numpy(n.reshape(w.n_req, w.n_kv_head)).cuda())

    sos = torch.zeros((w.n_req, w.n_kv_head, 8), dtype=torch.int32, device="cuda")
    stats = torch.zeros((2, 7), dtype=torch.int64, device="cuda")
    n_pf = n_pfh = 0
    for step in range(25):
        hs, hn = dev_sel([hints[u][step] for u in range(U)])
        g.ctx.layer_prefetch(1, hs, hn, g.ctx_len, stats)
        pfs = [layer_prefetch(caches[u], hints[u][step], 12 - 8) for u in range(U)]
        n_pf += sum(len(p.blocks) for p in pfs)
        _check_state(g, 1, caches, lens)
        _check_slots(g, 1, caches, lens, {u: pfs[u].blocks for u in range(U)})
        ss, sn = dev_sel([sels[u][step] for u in range(U)])
        g.ctx.cache_update(1, ss, sn, g.ctx_len, sos, stats)
        for u in range(U):
            n_pfh += cache_update(caches[u], sels[u][step]).prefetch_hits
        _check_state(g, 1, caches, lens)
    st = stats.cpu().numpy()[1]
    assert st[3] == n_pf and st[4] == n_pfh and n_pf > 0
    assert g.ctx.poll_error() == 0


@pytest.mark.parametrize("w,lens", [(TINY3, [4096, 1000, 17]), (TINY_G8, [4096, 3001]), (TINY_BS64, [3000, 2999]),
                                    (W.TINY_MLA, [4096]), (MLA_G128, [2048, 1999]), (MLA_G64, [2048, 1999]),
                                    (MLA_G128.with_(name="mla_g128_ragged", budget_blocks=700, cap_blocks=800), [2048, 777]),
                                    # one split (output written directly, no cluster) and three splits
                                    # (a cluster of 3: heads 43 / 43 / 42 per merging CTA)
                                    (MLA_G128.with_(name="mla_g128_one_split", budget_blocks=64, cap_blocks=128),
                                     [2048, 1500]),
                                    (MLA_G128.with_(name="mla_g128_three_splits", budget_blocks=200, cap_blocks=256),
                                     [2048, 999]),
                                    (MLA_G128_B8, [4096, 4000, 3001, 2048, 2047, 1500, 4096, 3333]),
                                    (W.TINY.with_(name="tiny_bigbudget", n_req=2, budget_blocks=300, cap_blocks=300),
                                     [4096, 4000]),
                                    (TINY3_FP8, [4096, 1000, 17]), (TINY_G8.with_(kv_dtype="fp8", v_scale=2.0), [4096, 3001])])
def test_sparse_decode_attention(w, lens):
    g = GpuCase(w, lens)
    U = g.ctx.units
    Kb = w.budget_blocks
    rng = np.random.default_rng(5)
    sel_h = np.zeros((U, Kb), np.int32)
    n_h = np.zeros(U, np.int32)
    sels = []
    for u in range(U):
        nb = _nb(lens[u // w.n_kv_head], w.block_size)
        k = min(Kb, nb)
        s = np.sort(np.concatenate([[nb - 1], rng.choice(nb - 1, k - 1, replace=False)])) if k > 1 else np.array([nb - 1])
        sels.append(s)
        sel_h[u, :k] = s
        n_h[u] = k
    sel = torch.from_numpy(sel_h.reshape(w.n_req, w.n_kv_head, Kb)).cuda()
    nsel = torch.from_numpy(n_h.reshape(w.n_req, w.n_kv_head)).cuda()
    sos = torch.zeros_like(sel)
    g.ctx.cache_update(0, sel, nsel, g.ctx_len, sos)
    q, _, _, _ = g.step_inputs(0)
    out = torch.zeros((w.n_req, w.n_q_head, w.d_v), dtype=torch.float32, device="cuda")
    g.ctx.sparse_decode_attn(0, _dev(q[0]), sel, sos, nsel, g.ctx_len, out)
    got = out.cpu().numpy()
    worst = 0.0
    for u in range(U):
        r, h = divmod(u, w.n_kv_head)
        L = lens[r]
        pos = np.concatenate([np.arange(b * w.block_size, min((b + 1) * w.block_size, L)) for b in sels[u]])
        kt = g.k_np[0, r, h, pos]
        vt = kt[:, : w.d_v] if w.v_shares_k else g.v_np[0, r, h, pos]
        if w.kv_dtype == "fp8":
            from oracle.fp8 import e4m3_decode
            kt, vt = e4m3_decode(kt) * float(w.k_scale), e4m3_decode(vt) * float(w.v_scale)
        heads = slice(h * w.group, (h + 1) * w.group)
        ref = attend(q[0, r, heads], kt, vt, w.softmax_scale)
        err = np.abs(got[r, heads] - ref).max()
        worst = max(worst, err)
        assert err <= 2e-3, f"unit {u}: max abs err {err}"
    assert g.ctx.poll_error() == 0


def test_append_rejects_misaligned_token_rows():
    """The appended rows are moved as 16-byte vectors: a misaligned k_new / v_new is refused on the
    host (KVS_ERR_INVALID_ARG) before anything is launched."""
    import sparse_kv_cache_decode_gb300 as K
    w = W.TINY_APPEND
    g = GpuCase(w, [w.ctx0])
    n = w.n_req * w.n_kv_head * w.d_k
    buf = torch.zeros(2 * n + 16, dtype=torch.int16, device="cuda")
    good_k, good_v = buf[:n], buf[n + 8:2 * n + 8]
    bad_k = buf[1:n + 1]                                   # 2 bytes past a 16-byte boundary
    for kk, vv in ((bad_k, good_v), (good_k, buf[n + 9:2 * n + 9])):
        with pytest.raises(K.KvsError) as e:
            g.ctx.append(0, kk, vv, g.index, g.ctx_len)
        assert K.STATUS[e.value.status] == "KVS_ERR_INVALID_ARG"
    torch.cuda.synchronize()
    assert g.ctx.poll_error() == 0


def test_quantize_e4m3_bit_exact():
    """kvs_quantize_e4m3 against the oracle's E4M3 encoder (round to nearest even, saturating):
    N(0, 1) and wide values, values near the subnormal range, exact ties, +-0 and beyond +-448."""
    import sparse_kv_cache_decode_gb300 as K
    from oracle import bf16_to_f32, f32_to_bf16_rne
    from oracle.fp8 import e4m3_encode
    rng = np.random.default_rng(21)
    x = np.concatenate([rng.normal(size=50001), rng.normal(size=20000) * 200, rng.normal(size=20000) * 0.004,
                        [0.0, -0.0, 448.0, 460.0, 470.0, -1e4, 17.0, 19.0, 248.0, 2.0 ** -10, 3 * 2.0 ** -10]])
    xb = f32_to_bf16_rne(x.astype(np.float32))
    for scale in (1.0, 0.5, 3.0):
        src = torch.from_numpy(xb.view(np.int16)).cuda()
        dst = torch.zeros(xb.size, dtype=torch.uint8, device="cuda")
        K.quantize_e4m3(src, dst, scale)
        torch.cuda.synchronize()
        ref = e4m3_encode((bf16_to_f32(xb) / np.float32(scale)).astype(np.float32))
        np.testing.assert_array_equal(dst.cpu().numpy(), ref, err_msg=f"scale {scale}")


def test_fp8_history_quantised_like_the_oracle():
    """The E4M3 history the library quantised equals the oracle's own encoding of the same values."""
    g = GpuCase(TINY3_FP8, [4096, 1000, 17])
    np.testing.assert_array_equal(g.k_host.numpy(), g.k_np)
    np.testing.assert_array_equal(g.v_host.numpy(), g.v_np)
