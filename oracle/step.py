"""One decode step over all layers, composed from the stage oracles (oracle; test-only).

Per step, layers in order; per (request, kv-head) unit of a layer:
  append (when tokens are given): the request's length L grows by one before layer 0; the new
      (k, v) is written at position L - 1 and the last block's index key is recomputed
      from its present tokens (the KV cache grows by one token per decode step: tuntang.top
      survey, introduction).
  prefetch (when enabled, layers > 0): the unit's cache takes the selection its request and
      kv-head made in the layer below as a hint (HiSparse page, insight 3).
  sync mode: score with the current query's group rows, select S_t, update (no pins), attend
      over S_t.
  lookahead mode (tuntang.top survey, section 3 step 1 pseudo-code; OasisKV page, key modules
      1-3): attend with the current query over S_t, the selection made in the previous step;
      score with the draft queries' group rows, select S_{t+1}, update with S_t pinned.  The
      first step has no S_t yet and bootstraps it in sync mode from the current query.
Lookahead mode is defined without append and without prefetch (those combinations are not
part of this build's workloads).  With w.evict_policy == "importance" every update evicts the
least important blocks by the scores that made its selection (see oracle.cache).  snapshot() and
restore() save and put back every unit's cache state and pending selection (speculative
rollback, KV-cache overview, section 6.1).  With w.score_mode == "bound" blocks are summarised by
their per-dimension [max | min] keys and scored by the query-aware upper bound (oracle.bound)
instead of the block-mean key.  With w.kv_dtype == "fp8" the history holds E4M3 codes (oracle.fp8):
keys and values are decode(code) * k_scale / v_scale, the index keys sum their fp32 values, and an
appended token is quantised on arrival.

Parity-relevant outputs are recorded per unit (UnitRecord) and per layer (stats()).
"""
from dataclasses import dataclass

import numpy as np

from .attention import attend
from .bound import block_scores_bound, index_minmax, index_minmax_block
from .bf16 import bf16_to_f32
from .fp8 import dequantize_f32, e4m3_decode, quantize
from .cache import PrefetchResult, UnitCache, UpdateResult, cache_restore, cache_update, layer_prefetch
from .index_keys import index_key_block, index_keys
from .scores import block_scores
from .select import select_blocks


@dataclass
class UnitRecord:
    attn_sel: np.ndarray      # blocks the attention read in this step
    sel: np.ndarray           # selection made in this step (S_t in sync mode, S_{t+1} in lookahead)
    scores: np.ndarray        # fp32 block scores behind `sel`
    bound: np.ndarray         # A[b] behind `scores` (fp64)
    update: UpdateResult      # the update that made `sel` resident
    boot: tuple = None        # lookahead first step: (scores, bound, sel, update) of the sync part
    prefetch: PrefetchResult = None
    ctx_len: int = 0


class OracleDecoder:
    def __init__(self, w, host_k, host_v, ctx_len, reqs=None):
        """host_k[l, r, h] -> (>= max_ctx, d_k) bf16 rows (likewise host_v, or None for MLA).
        Rows of the requests in `reqs` are copied, so later writes to host_k do not leak in."""
        if w.lookahead and (w.append or w.layer_prefetch):
            raise ValueError("lookahead mode is defined without append and without prefetch")
        self.w = w
        self.bound = getattr(w, "score_mode", "mean") == "bound"
        self.fp8 = getattr(w, "kv_dtype", "bf16") == "fp8"
        if self.fp8 and (self.bound or w.v_shares_k):
            raise ValueError("FP8 history is defined for block-mean scoring of separate K and V")
        self.reqs = list(range(w.n_req)) if reqs is None else list(reqs)
        self.L = {r: int(ctx_len[r]) for r in self.reqs}
        self.k, self.v, self.ik, self.cache, self.pending = {}, {}, {}, {}, {}
        for l in range(w.n_layer):
            for r in self.reqs:
                for h in range(w.n_kv_head):
                    u = (l, r, h)
                    self.k[u] = np.array(host_k[l, r, h][: w.max_ctx], copy=True)
                    self.v[u] = None if w.v_shares_k else np.array(host_v[l, r, h][: w.max_ctx], copy=True)
                    nb = self.n_blocks(r)
                    if self.bound:
                        ik = np.zeros((w.max_blocks, 2 * w.d_k), np.uint16)
                        ik[:nb] = index_minmax(self.k[u], self.L[r], w.block_size)
                    else:
                        ik = np.zeros((w.max_blocks, w.d_k), np.uint16)
                        ik[:nb] = index_keys(self.key_values(u), self.L[r], w.block_size)
                    self.ik[u] = ik
                    self.cache[u] = UnitCache(w.cap_blocks, w.max_blocks)
                    self.pending[u] = None
        self.max_prefetch = w.cap_blocks - w.budget_blocks
        self.records = {}

    def n_blocks(self, r: int) -> int:
        return (self.L[r] + self.w.block_size - 1) // self.w.block_size

    def row_bytes(self) -> int:
        w = self.w
        return (1 if self.fp8 else 2) * (w.d_k + (0 if w.v_shares_k else w.d_v))

    def key_values(self, u, rows=slice(None)):
        """Key rows for the index: bf16 patterns, or fp32 values of FP8 codes."""
        k = self.k[u][rows]
        return dequantize_f32(k, self.w.k_scale) if self.fp8 else k

    def tokens(self, u, sel):
        w, (l, r, h) = self.w, u
        bs, L = w.block_size, self.L[r]
        if len(sel) == 0:
            pos = np.zeros(0, np.int64)
        else:
            pos = np.concatenate([np.arange(b * bs, min((b + 1) * bs, L)) for b in sel])
        k = self.k[u][pos]
        v = k[:, : w.d_v] if w.v_shares_k else self.v[u][pos]
        if self.fp8:
            k = e4m3_decode(k) * float(w.k_scale)
            v = e4m3_decode(v) * float(w.v_scale)
        return k, v

    def _score_select(self, u, rows):
        w, r = self.w, u[1]
        nb = self.n_blocks(r)
        score = block_scores_bound if self.bound else block_scores
        s64, a = score(rows, self.ik[u][:nb], w.softmax_scale)
        s32 = s64.astype(np.float32)
        sel = select_blocks(s32, nb, w.budget_blocks, w.n_sink, w.n_recent)
        return s32, a, sel

    def _append(self, u, k_new, v_new):
        w, r = self.w, u[1]
        p = self.L[r] - 1
        if self.fp8:
            k_new = quantize(bf16_to_f32(k_new), w.k_scale)
            v_new = quantize(bf16_to_f32(v_new), w.v_scale)
        self.k[u][p] = k_new
        if not w.v_shares_k:
            self.v[u][p] = v_new
        b = p // w.block_size
        summarise = index_minmax_block if self.bound else index_key_block
        self.ik[u][b] = summarise(self.key_values(u, slice(b * w.block_size, self.L[r])))

    def step(self, q, score_q=None, new_k=None, new_v=None):
        """q: [N_l][B][H_q][D_k] bf16; score_q: [N_l][B][n_draft][H_q][D_k] drafts (lookahead);
        new_k / new_v: [N_l][B][H_kv][D] appended tokens or None.
        Returns out [N_l][len(reqs)][H_q][D_v] fp32 and {(l, r, h): UnitRecord}."""
        w = self.w
        g = w.group
        if new_k is not None:
            for r in self.reqs:
                self.L[r] += 1
        out = np.zeros((w.n_layer, len(self.reqs), w.n_q_head, w.d_v), np.float32)
        recs = {}
        for l in range(w.n_layer):
            for ri, r in enumerate(self.reqs):
                for h in range(w.n_kv_head):
                    u = (l, r, h)
                    if new_k is not None:
                        self._append(u, new_k[l, r, h], None if w.v_shares_k else new_v[l, r, h])
                    pf = None
                    if w.layer_prefetch and l > 0:
                        pf = layer_prefetch(self.cache[u], recs[(l - 1, r, h)].sel, self.max_prefetch)
                    heads = slice(h * g, (h + 1) * g)
                    qh = q[l, r, heads]
                    boot = None
                    imp = getattr(w, "evict_policy", "lru") == "importance"
                    if not w.lookahead:
                        s32, a, sel = self._score_select(u, qh)
                        upd = cache_update(self.cache[u], sel, importance=s32 if imp else None)
                        attn_sel = sel
                    else:
                        attn_sel = self.pending[u]
                        if attn_sel is None:
                            b32, ba, bsel = self._score_select(u, qh)
                            bupd = cache_update(self.cache[u], bsel, importance=b32 if imp else None)
                            boot = (b32, ba, bsel, bupd)
                            attn_sel = bsel
                        rows = score_q[l, r, :, heads].reshape(-1, w.d_k)
                        s32, a, sel = self._score_select(u, rows)
                        upd = cache_update(self.cache[u], sel, pinned=attn_sel, importance=s32 if imp else None)
                        self.pending[u] = sel
                    kt, vt = self.tokens(u, attn_sel)
                    out[l, ri, heads] = attend(qh, kt, vt, w.softmax_scale)
                    recs[u] = UnitRecord(attn_sel, sel, s32, a, upd, boot, pf, self.L[r])
        self.records = recs
        return out, recs

    def snapshot(self, layer=None):
        """Copies of the cache state and pending selection of every unit (of one layer)."""
        return {u: (c.copy(), None if self.pending[u] is None else self.pending[u].copy())
                for u, c in self.cache.items() if layer is None or u[0] == layer}

    def restore(self, snap):
        """Put the units of a snapshot back; returns {unit: (slots, blocks)} to fetch again."""
        out = {}
        for u, (c, pend) in snap.items():
            out[u] = cache_restore(self.cache[u], c)
            self.pending[u] = None if pend is None else pend.copy()
        return out

    def fetched_rows(self, r: int, blocks) -> int:
        bs, L = self.w.block_size, self.L[r]
        return int(sum(min(bs, L - b * bs) for b in blocks))

    def stats(self, recs=None, layer=None) -> dict:
        """Per-layer counters of the last step: hits, misses, evictions, prefetched,
        prefetch_hits, pin_fallbacks, bytes_fetched (misses and prefetches, rows < L)."""
        recs = self.records if recs is None else recs
        out = {}
        for (l, r, h), rec in recs.items():
            if layer is not None and l != layer:
                continue
            st = out.setdefault(l, dict(hits=0, misses=0, evictions=0, prefetched=0, prefetch_hits=0,
                                        pin_fallbacks=0, bytes_fetched=0))
            updates = [rec.update] + ([rec.boot[3]] if rec.boot is not None else [])
            for upd in updates:
                st["hits"] += len(upd.hits)
                st["misses"] += len(upd.misses)
                st["evictions"] += upd.n_evictions
                st["prefetch_hits"] += upd.prefetch_hits
                st["pin_fallbacks"] += int(upd.pin_fallback)
                st["bytes_fetched"] += self.fetched_rows(r, upd.misses) * self.row_bytes()
            if rec.prefetch is not None:
                st["prefetched"] += len(rec.prefetch.blocks)
                st["evictions"] += int((rec.prefetch.evicted >= 0).sum())
                st["bytes_fetched"] += self.fetched_rows(r, rec.prefetch.blocks) * self.row_bytes()
        return out
