"""Shared set-up for the GPU parity tests: one workload bound to a libkvs context, and the
oracle on the same seeded inputs.  Inputs only ever flow oracle/generator -> GPU; the oracle
never reads anything the CUDA path wrote."""
from __future__ import annotations

import math

import numpy as np

import workload as W
from oracle import OracleDecoder, bf16_to_f32


def torch_mod():
    import torch
    return torch


class GpuCase:
    """Host history (pinned), device index, contexts and per-step buffers for one workload."""

    def __init__(self, w: W.Workload, ctx_lens=None, copy_stream=False, n_threads=0):
        torch = torch_mod()
        import sparse_kv_cache_decode_gb300 as K
        self.w = w
        self.K = K
        B, NL, Hkv = w.n_req, w.n_layer, w.n_kv_head
        kshape = (NL, B, Hkv, w.max_ctx, w.d_k)
        vshape = None if w.v_shares_k else (NL, B, Hkv, w.max_ctx, w.d_v)
        self._arrays = []
        self.k_bf16 = self.v_bf16 = None
        if getattr(w, "kv_dtype", "bf16") == "fp8":
            # E4M3 history: the library quantises the generator's bf16 values on the GPU; the oracle
            # quantises the same values with its own encoder (tests compare the two code arrays)
            from oracle import bf16_to_f32
            from oracle.fp8 import quantize
            kb = torch.empty(kshape, dtype=torch.int16, pin_memory=True)
            vb = torch.empty(vshape, dtype=torch.int16, pin_memory=True)
            W.fill_kv(w, kb, vb, n_threads)
            self.k_host = torch.empty(kshape, dtype=torch.uint8, pin_memory=True)
            self.v_host = torch.empty(vshape, dtype=torch.uint8, pin_memory=True)
            K.quantize_history_e4m3(kb, self.k_host, w.k_scale)
            K.quantize_history_e4m3(vb, self.v_host, w.v_scale)
            self.k_bf16, self.v_bf16 = kb.numpy().view(np.uint16), vb.numpy().view(np.uint16)
            self.k_np = quantize(bf16_to_f32(self.k_bf16), w.k_scale)
            self.v_np = quantize(bf16_to_f32(self.v_bf16), w.v_scale)
        elif w.host_kv_bytes >= (1 << 30):
            # large histories: huge-page host arrays, released by close() (torch keeps freed
            # pinned blocks cached, which would exhaust host memory across full-size tests)
            ka = K.HostArray(kshape)
            va = None if vshape is None else K.HostArray(vshape)
            self.k_host, self.v_host = ka.tensor, None if va is None else va.tensor
            W.fill_kv(w, self.k_host, self.v_host, n_threads)
            ka.register()
            if va is not None:
                va.register()
            self._arrays = [a for a in (ka, va) if a is not None]
        else:
            self.k_host = torch.empty(kshape, dtype=torch.int16, pin_memory=True)
            self.v_host = None if vshape is None else torch.empty(vshape, dtype=torch.int16, pin_memory=True)
            W.fill_kv(w, self.k_host, self.v_host, n_threads)
        if self.k_bf16 is None:
            self.k_np = self.k_host.numpy().view(np.uint16)
            self.v_np = None if self.v_host is None else self.v_host.numpy().view(np.uint16)
        self.ctx_lens = list(ctx_lens) if ctx_lens is not None else [w.ctx0] * B
        self.ctx_len = torch.tensor(self.ctx_lens, dtype=torch.int32, device="cuda")
        self.cfg = K.make_config(w)
        self.ctx = K.Context(self.cfg)
        self.ctx.bind_host_kv(self.k_host, self.v_host)
        self.nb_max = w.max_blocks
        self.index = torch.zeros((NL, B, Hkv, self.nb_max, w.d_idx), dtype=torch.int16, device="cuda")
        for l in range(NL):
            self.ctx.index_build(l, self.index, self.ctx_len)
        self.stats = torch.zeros((NL, 7), dtype=torch.int64, device="cuda")
        self.sel = torch.zeros((NL, B, Hkv, w.budget_blocks), dtype=torch.int32, device="cuda")
        self.nsel = torch.zeros((NL, B, Hkv), dtype=torch.int32, device="cuda")
        self.out = torch.zeros((NL, B, w.n_q_head, w.d_v), dtype=torch.float32, device="cuda")
        self.copy_stream = torch.cuda.Stream() if copy_stream else None
        self.qs = W.QueryStream(w)
        self.t = 0
        torch.cuda.synchronize()

    def close(self):
        """Release the context and the host history now (full-size cases hold tens of GiB)."""
        import gc
        torch = torch_mod()
        torch.cuda.synchronize()
        self.ctx.close()
        for a in self._arrays:
            a.close()
        self._arrays = []
        self.k_host = self.v_host = self.k_np = self.v_np = None
        gc.collect()

    def oracle(self, reqs=None) -> OracleDecoder:
        """Oracle on the same inputs (copies the host rows now, before any GPU append)."""
        return OracleDecoder(self.w, self.k_np, self.v_np, self.ctx_lens, reqs)

    def step_inputs(self, t: int):
        w = self.w
        q = self.qs.queries(t)
        d = self.qs.drafts(t) if w.lookahead else None
        nk = nv = None
        if w.append:
            nk, nv = W.token(w, w.ctx0 + t)
        return q, d, nk, nv

    def gpu_step(self, q, d, nk, nv):
        """One decode step over all layers through kvs_decode_step (+ prefetch, append)."""
        torch = torch_mod()
        w = self.w
        qd = torch.from_numpy(q.view(np.int16)).cuda()
        dd = None if d is None else torch.from_numpy(d.view(np.int16)).cuda()
        nkd = None if nk is None else torch.from_numpy(nk.view(np.int16)).cuda()
        nvd = None if nv is None else torch.from_numpy(nv.view(np.int16)).cuda()
        if w.append:
            self.ctx.advance_ctx(self.ctx_len)
        for l in range(w.n_layer):
            if w.layer_prefetch and l > 0:
                self.ctx.layer_prefetch(l, self.sel[l - 1], self.nsel[l - 1], self.ctx_len, self.stats,
                                        stream=self.copy_stream)
            self.ctx.decode_step(l, qd[l], None if dd is None else dd[l], w.n_score_q if dd is not None else 1,
                                 self.index, self.ctx_len, self.out[l], self.stats,
                                 None if nkd is None else nkd[l], None if nvd is None else nvd[l],
                                 self.sel[l], self.nsel[l], copy_stream=self.copy_stream)
        self.ctx.join()
        torch.cuda.synchronize()
        self.t += 1


def score_tolerance(s_ref: np.ndarray, a_ref: np.ndarray) -> np.ndarray:
    """|s_gpu - s| <= 1e-4 (|s| + A): the relative 1e-4 score bound, measured against the
    conditioning A = scale * max sum |q.ik| so that near-cancelling dot products are fair."""
    return 1e-4 * (np.abs(s_ref) + a_ref)


def selection_is_valid(sel, s_ref, a_ref, nb, budget, n_sink, n_recent) -> bool:
    """A GPU selection that differs from the oracle's is still correct when some perturbation
    of the reference scores within the tolerance makes it the top-K (several results are
    correct at near-ties): every chosen free block must not lose to an unchosen one by more
    than the two tolerances."""
    from oracle import forced_blocks
    sel = np.asarray(sel)
    if nb <= budget:
        return sel.tolist() == list(range(nb))
    forced = set(forced_blocks(nb, budget, n_sink, n_recent).tolist())
    if not forced <= set(sel.tolist()) or len(sel) != budget or np.any(np.diff(sel) <= 0):
        return False
    tol = score_tolerance(s_ref, a_ref)
    chosen = [b for b in sel if b not in forced]
    rest = np.array([b for b in range(nb) if b not in forced and b not in set(chosen)], np.int64)
    if len(rest) == 0:
        return True
    worst_chosen = min(s_ref[b] + tol[b] for b in chosen)
    best_rest = np.max(s_ref[rest] - tol[rest])
    return worst_chosen >= best_rest


STAT_KEYS = ["hits", "misses", "evictions", "prefetched", "prefetch_hits", "pin_fallbacks", "bytes_fetched"]


def compare_step(g, o, out_ref, recs, cum, exact=True, frozen=None):
    """Compare one GPU step with the oracle's on the oracle's requests: selection, cache state
    and attention output per unit.  exact: selections must match (and per-layer counters, when
    the oracle covers every request).  Otherwise a differing selection must be a valid top-K under
    the score tolerance (a near tie), and that unit is frozen (its state diverges from then on)."""
    w = g.w
    sel = g.sel.cpu().numpy()
    nsel = g.nsel.cpu().numpy()
    out = g.out.cpu().numpy()
    for l in range(w.n_layer):
        b2s, s2b, st, clk = g.ctx.cache_export(l)
        for ri, r in enumerate(o.reqs):
            for h in range(w.n_kv_head):
                u = r * w.n_kv_head + h
                rec = recs[(l, r, h)]
                heads = slice(h * w.group, (h + 1) * w.group)
                if frozen is not None and (l, r, h) in frozen:
                    continue
                if frozen is not None and w.layer_prefetch and (l - 1, r, h) in frozen:
                    frozen.add((l, r, h))      # its prefetch hint came from a diverged layer
                    continue
                got_sel = sel[l, r, h, : nsel[l, r, h]]
                same = got_sel.tolist() == rec.sel.tolist()
                if not same:
                    assert not exact, f"layer {l} unit {(r, h)}: selection differs"
                    nb = o.n_blocks(r)
                    assert selection_is_valid(got_sel, rec.scores.astype(np.float64), rec.bound, nb,
                                              w.budget_blocks, w.n_sink, w.n_recent), f"invalid selection {(l, r, h)}"
                    frozen.add((l, r, h))
                    continue
                c = o.cache[(l, r, h)]
                np.testing.assert_array_equal(s2b[u], c.slot2block, err_msg=f"slot2block {(l, r, h)}")
                np.testing.assert_array_equal(st[u].astype(np.int64), c.stamp, err_msg=f"stamp {(l, r, h)}")
                assert int(clk[u]) == c.clock
                err = np.abs(out[l, r, heads] - out_ref[l, ri, heads]).max()
                assert err <= 2e-3, f"layer {l} unit {(r, h)}: attention max abs err {err}"
    if exact:
        st_ref = o.stats(recs)
        for l in range(w.n_layer):
            for k in STAT_KEYS:
                cum[l][k] += st_ref[l][k]
        got = g.stats.cpu().numpy()
        for l in range(w.n_layer):
            assert [int(x) for x in got[l]] == [cum[l][k] for k in STAT_KEYS], f"stats layer {l}"
