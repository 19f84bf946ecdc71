"""Pins for oracle.step: dense equivalence (torch SDPA), append, prefetch and lookahead properties."""
import math

import numpy as np
import pytest
import torch

import workload as W
from oracle import OracleDecoder, bf16_to_f32, index_keys


def _sdpa(q_rows, k_tok, v_tok, scale):
    g = q_rows.shape[0]
    tq = torch.from_numpy(bf16_to_f32(q_rows).astype(np.float64))[None, :, None, :]
    tk = torch.from_numpy(bf16_to_f32(k_tok).astype(np.float64))[None, None].expand(1, g, -1, -1)
    tv = torch.from_numpy(bf16_to_f32(v_tok).astype(np.float64))[None, None].expand(1, g, -1, -1)
    return torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)[0, :, 0].numpy()


SMALL = W.TINY.with_(name="small", ctx0=1000, steps=4, budget_blocks=8, cap_blocks=12, n_heavy=8)


def test_budget_covering_context_is_dense_attention():
    w = SMALL.with_(budget_blocks=64, cap_blocks=64)      # 1000 tokens = 63 blocks <= 64
    k, v = W.kv_numpy(w)
    dec = OracleDecoder(w, k, v, [w.ctx0])
    qs = W.QueryStream(w)
    for t in range(3):
        q = qs.queries(t)
        out, recs = dec.step(q)
        for h in range(w.n_kv_head):
            heads = slice(h * w.group, (h + 1) * w.group)
            ref = _sdpa(q[0, 0, heads], k[0, 0, h, : w.ctx0], v[0, 0, h, : w.ctx0], w.softmax_scale)
            np.testing.assert_allclose(out[0, 0, heads], ref, atol=1e-6, rtol=0)
            assert recs[(0, 0, h)].sel.tolist() == list(range(63))


def test_each_request_and_layer_attends_over_its_own_tokens():
    """Two layers and two requests of different lengths (1000 and 517 tokens: 63 and 33 blocks,
    budget 64): each (layer, request) output is dense attention over that layer's and request's
    own tokens only."""
    w = SMALL.with_(name="two_req", n_req=2, n_layer=2, budget_blocks=64, cap_blocks=64)
    k, v = W.kv_numpy(w)
    lens = [1000, 517]
    dec = OracleDecoder(w, k, v, lens)
    q = W.QueryStream(w).queries(0)
    out, recs = dec.step(q)
    for l in range(2):
        for r, n in enumerate(lens):
            for h in range(w.n_kv_head):
                heads = slice(h * w.group, (h + 1) * w.group)
                ref = _sdpa(q[l, r, heads], k[l, r, h, :n], v[l, r, h, :n], w.softmax_scale)
                np.testing.assert_allclose(out[l, r, heads], ref, atol=1e-6, rtol=0)
                assert recs[(l, r, h)].sel.tolist() == list(range((n + 15) // 16))


def test_mla_budget_covering_context_is_dense_attention_over_the_latent():
    """MLA reading: every q head attends over the full latent row as K and its first d_v entries
    as V (one latent head shared by all 16 q heads); with the budget above the context the step is
    dense attention, so a wrong value slice, head mapping or scale fails here."""
    w = W.TINY_MLA.with_(name="mla_dense", ctx0=200, steps=3)            # bs 1: 200 blocks <= K_b 256
    k, _ = W.kv_numpy(w)
    dec = OracleDecoder(w, k, None, [w.ctx0])
    qs = W.QueryStream(w)
    assert w.softmax_scale == float(np.float32(1.0 / 24.0))             # 1 / sqrt(576), held in fp32
    for t in range(2):
        q = qs.queries(t)
        out, recs = dec.step(q)
        lat = k[0, 0, 0, : w.ctx0]
        ref = _sdpa(q[0, 0], lat, lat[:, : w.d_v], w.softmax_scale)
        assert out.shape[-1] == 512
        np.testing.assert_allclose(out[0, 0], ref, atol=1e-6, rtol=0)
        assert recs[(0, 0, 0)].sel.tolist() == list(range(w.ctx0))


def _brute_selection(rows, ik, nb, budget, n_sink, n_recent, scale):
    """Sink + recent + the best of the rest, each block scored as the largest scaled dot product
    over the given query rows (exact sums), ties to the lower block; ascending block ids."""
    rows64 = [bf16_to_f32(r).astype(np.float64) for r in rows]
    keys64 = [bf16_to_f32(k).astype(np.float64) for k in ik]
    score = [np.float32(scale * max(math.fsum(a * b for a, b in zip(r, keys64[blk])) for r in rows64))
             for blk in range(nb)]
    if nb <= budget:
        return list(range(nb))
    forced = set(range(min(n_sink, nb))) | set(range(max(0, nb - n_recent), nb))
    rest = sorted((blk for blk in range(nb) if blk not in forced), key=lambda blk: (-score[blk], blk))
    return sorted(forced | set(rest[: budget - len(forced)]))


@pytest.mark.parametrize("lookahead", [False, True])
def test_selection_scores_each_kv_head_with_its_own_group_and_every_draft(lookahead):
    """Scoring rows of kv head h are q heads [h G, (h + 1) G) (contiguous groups), and in lookahead
    mode those heads of every draft; checked against a brute-force selection on a ragged 300-token
    context (19 blocks, budget 8 = 1 sink + 2 recent + 5 scored)."""
    base = W.TINY_LOOKAHEAD if lookahead else W.TINY
    w = base.with_(name="sel_rows", ctx0=300, steps=3, budget_blocks=8, cap_blocks=12)
    k, v = W.kv_numpy(w)
    dec = OracleDecoder(w, k, v, [w.ctx0])
    qs = W.QueryStream(w)
    g, nb = w.group, 19
    for t in range(2):
        q = qs.queries(t)
        d = qs.drafts(t) if lookahead else None
        _, recs = dec.step(q, d)
        for h in range(w.n_kv_head):
            ik = index_keys(k[0, 0, h], w.ctx0, w.block_size)
            if lookahead:
                rows = [d[0, 0, j, hq] for j in range(w.n_draft) for hq in range(h * g, (h + 1) * g)]
            else:
                rows = [q[0, 0, hq] for hq in range(h * g, (h + 1) * g)]
            want = _brute_selection(rows, ik, nb, w.budget_blocks, w.n_sink, w.n_recent, w.softmax_scale)
            assert recs[(0, 0, h)].sel.tolist() == want, (t, h)


def test_ragged_tail_and_capacity_do_not_change_outputs():
    w = SMALL.with_(ctx0=1000)
    k, v = W.kv_numpy(w)
    qs1, qs2 = W.QueryStream(w), W.QueryStream(w)
    d1 = OracleDecoder(w, k, v, [997])                               # ragged: 997 = 62*16 + 5
    d2 = OracleDecoder(w.with_(cap_blocks=40), k, v, [997])
    for t in range(4):
        o1, r1 = d1.step(qs1.queries(t))
        o2, r2 = d2.step(qs2.queries(t))
        np.testing.assert_array_equal(o1, o2)
        for u in r1:
            assert r1[u].sel.tolist() == r2[u].sel.tolist()
            assert max(r1[u].sel) <= 62


def test_append_updates_last_block_key_and_length():
    w = SMALL.with_(append=True, ctx0=1000, steps=20)
    k, v = W.kv_numpy(w)
    dec = OracleDecoder(w, k, v, [w.ctx0])
    qs = W.QueryStream(w)
    full_k = k.copy()
    for t in range(20):
        nk, nv = W.token(w, w.ctx0 + t)
        full_k[:, :, :, w.ctx0 + t] = nk
        dec.step(qs.queries(t), new_k=nk, new_v=nv)
        L = w.ctx0 + t + 1
        assert dec.L[0] == L
        for h in range(w.n_kv_head):
            nb = (L + 15) // 16
            np.testing.assert_array_equal(dec.ik[(0, 0, h)][:nb], index_keys(full_k[0, 0, h], L, 16))
            # the recent blocks (which hold the new token) are always selected
            assert nb - 1 in dec.records[(0, 0, h)].sel


def test_query_attends_to_the_token_appended_with_it():
    """Reading 14: the query of a step attends to [0, L) after that step's append, its own token
    included; with the budget above the context the output is dense attention over all of them."""
    w = SMALL.with_(name="append_dense", append=True, ctx0=1000, steps=4, budget_blocks=64, cap_blocks=64)
    k, v = W.kv_numpy(w)
    dec = OracleDecoder(w, k, v, [w.ctx0])
    qs = W.QueryStream(w)
    full_k, full_v = k.copy(), v.copy()
    for t in range(3):
        nk, nv = W.token(w, w.ctx0 + t)
        full_k[:, :, :, w.ctx0 + t], full_v[:, :, :, w.ctx0 + t] = nk, nv
        q = qs.queries(t)
        out, _ = dec.step(q, new_k=nk, new_v=nv)
        L = w.ctx0 + t + 1
        for h in range(w.n_kv_head):
            heads = slice(h * w.group, (h + 1) * w.group)
            ref = _sdpa(q[0, 0, heads], full_k[0, 0, h, :L], full_v[0, 0, h, :L], w.softmax_scale)
            np.testing.assert_allclose(out[0, 0, heads], ref, atol=1e-6, rtol=0)
            without = _sdpa(q[0, 0, heads], full_k[0, 0, h, : L - 1], full_v[0, 0, h, : L - 1], w.softmax_scale)
            assert np.abs(without - ref).max() > 1e-4        # the new token is not negligible here


def test_prefetch_never_changes_outputs():
    w = SMALL.with_(n_layer=3, layer_prefetch=True, rho_layer=0.8, cap_blocks=14)
    k, v = W.kv_numpy(w)
    a = OracleDecoder(w, k, v, [w.ctx0])
    b = OracleDecoder(w.with_(layer_prefetch=False), k, v, [w.ctx0])
    qa, qb = W.QueryStream(w), W.QueryStream(w)
    total_pf = 0
    for t in range(4):
        oa, ra = a.step(qa.queries(t))
        ob, rb = b.step(qb.queries(t))
        np.testing.assert_array_equal(oa, ob)
        for u, rec in ra.items():
            assert rec.sel.tolist() == rb[u].sel.tolist()
            if u[0] > 0:
                assert len(rec.prefetch.blocks) <= a.max_prefetch
                total_pf += len(rec.prefetch.blocks)
        st = a.stats()
        for l in st:
            assert st[l]["hits"] + st[l]["misses"] == sum(len(ra[u].sel) for u in ra if u[0] == l)
    assert total_pf > 0


def test_lookahead_pins_attention_set():
    w = SMALL.with_(lookahead=True, n_draft=4)
    k, v = W.kv_numpy(w)
    dec = OracleDecoder(w, k, v, [w.ctx0])
    qs = W.QueryStream(w)
    prev = None
    for t in range(5):
        out, recs = dec.step(qs.queries(t), qs.drafts(t))
        for u, rec in recs.items():
            if t == 0:
                assert rec.boot is not None
            else:
                assert rec.boot is None and rec.attn_sel.tolist() == prev[u].tolist()
            if not rec.update.pin_fallback:
                assert set(rec.attn_sel.tolist()) <= dec.cache[u].resident()
            assert set(rec.sel.tolist()) <= dec.cache[u].resident()
        prev = {u: rec.sel for u, rec in recs.items()}


def test_fp8_history_with_exact_values_matches_bf16():
    """Integer-valued keys and values (|x| <= 16) and power-of-two scales are exact in E4M3, so the
    FP8 decoder must reproduce the bf16 decoder exactly -- selections, cache state, outputs --
    with half the fetched bytes; an appended token is quantised on arrival."""
    from oracle import bf16_to_f32
    from oracle.fp8 import quantize
    w = SMALL.with_(int_scale=2.0, int_clip=4.0, append=True, steps=6)   # heavy keys up to 16: 2k <= 32, even
    w8 = w.with_(kv_dtype="fp8", k_scale=0.5, v_scale=2.0)
    k, v = W.kv_numpy(w)
    a = OracleDecoder(w, k, v, [w.ctx0])
    b = OracleDecoder(w8, quantize(bf16_to_f32(k), w8.k_scale), quantize(bf16_to_f32(v), w8.v_scale), [w.ctx0])
    qa, qb = W.QueryStream(w), W.QueryStream(w8)
    for t in range(6):
        nk, nv = W.token(w, w.ctx0 + t)
        oa, ra = a.step(qa.queries(t), new_k=nk, new_v=nv)
        ob, rb = b.step(qb.queries(t), new_k=nk, new_v=nv)
        np.testing.assert_array_equal(oa, ob)
        for u in ra:
            assert ra[u].sel.tolist() == rb[u].sel.tolist()
            np.testing.assert_array_equal(a.ik[u], b.ik[u])
        sa, sb = a.stats(), b.stats()
        assert sa[0]["bytes_fetched"] == 2 * sb[0]["bytes_fetched"]
        assert {k2: v2 for k2, v2 in sa[0].items() if k2 != "bytes_fetched"} == \
               {k2: v2 for k2, v2 in sb[0].items() if k2 != "bytes_fetched"}


def test_fp8_quantisation_error_is_bounded():
    """With N(0,1) values the FP8 decoder's outputs stay within E4M3's relative step (2^-4 of each
    value at most) of the bf16 decoder's: the dequantised rows differ by at most that much."""
    from oracle import bf16_to_f32
    from oracle.fp8 import dequantize_f32, quantize
    k, _ = W.kv_numpy(SMALL)
    x = bf16_to_f32(k)
    err = np.abs(dequantize_f32(quantize(x, 1.0), 1.0) - x)
    assert np.all(err <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10))
