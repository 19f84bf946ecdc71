"""Error paths through the C ABI, each made on the host with inputs the library's own checks turn
into a status (nothing here can fault the GPU: every bad index is validated before it is used):
  * out-of-range, unordered or over-long selections passed to kvs_cache_update -> device status
    KVS_ERR_BAD_INDEX, and the refused unit's cache state is left as it was;
  * out-of-range slots, block ids and counts passed to kvs_sparse_decode_attn (the TMA kernel and
    the cp.async kernel) -> KVS_ERR_BAD_INDEX, with every other unit's output unchanged;
  * host memory that is not page-locked and mapped -> KVS_ERR_HOST_MEM from kvs_bind_host_kv;
  * bad layers, widths and pointers -> KVS_ERR_INVALID_ARG before any launch.
A wait that runs out of time (KVS_ERR_TIMEOUT) is not provoked on the GPU."""
import numpy as np
import pytest

import workload as W
from kvs_harness import GpuCase

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

BAD_INDEX, INVALID_ARG, HOST_MEM = 7, 1, 5


def _first_blocks(g, n):
    w = g.w
    sel = torch.zeros((w.n_req, w.n_kv_head, w.budget_blocks), dtype=torch.int32, device="cuda")
    sel[..., :n] = torch.arange(n, dtype=torch.int32, device="cuda")
    nsel = torch.full((w.n_req, w.n_kv_head), n, dtype=torch.int32, device="cuda")
    return sel, nsel


@pytest.mark.parametrize("bad", ["past_end", "negative", "unordered", "duplicate", "count"])
def test_cache_update_refuses_bad_selection(bad):
    w = W.TINY.with_(name="err_update", n_req=2)
    g = GpuCase(w, [4096, 1000])
    sel, nsel = _first_blocks(g, 16)
    sos = torch.zeros_like(sel)
    g.ctx.cache_update(0, sel, nsel, g.ctx_len, sos, g.stats)          # a good update first
    torch.cuda.synchronize()
    assert g.ctx.poll_error() == 0
    b2s0, s2b0, st0, clk0 = g.ctx.cache_export(0)
    sel2 = sel + 20                                                     # blocks 20..35 (all misses)
    r, h = 1, 0                                                         # the unit made bad
    if bad == "past_end":
        sel2[r, h, 15] = (1000 + 15) // 16                              # one past its last block
    elif bad == "negative":
        sel2[r, h, 0] = -1
    elif bad == "unordered":
        sel2[r, h, 3], sel2[r, h, 4] = sel2[r, h, 4].item(), sel2[r, h, 3].item()
    elif bad == "duplicate":
        sel2[r, h, 5] = sel2[r, h, 4]
    else:
        nsel[r, h] = w.budget_blocks + 1
    g.ctx.cache_update(0, sel2, nsel, g.ctx_len, sos, g.stats)
    torch.cuda.synchronize()
    assert g.ctx.poll_error() == BAD_INDEX
    b2s1, s2b1, st1, clk1 = g.ctx.cache_export(0)
    u = r * w.n_kv_head + h
    np.testing.assert_array_equal(b2s1[u], b2s0[u])
    np.testing.assert_array_equal(s2b1[u], s2b0[u])
    np.testing.assert_array_equal(st1[u], st0[u])
    assert clk1[u] == clk0[u]
    others = [v for v in range(g.ctx.units) if v != u]
    assert all(clk1[v] == clk0[v] + 1 for v in others)                # the rest were accepted
    assert g.ctx.poll_error() == 0                                      # the word was cleared
    g.close()


@pytest.mark.parametrize("w", [W.TINY.with_(name="err_attn_tma", n_req=2),
                               W.TINY_MLA.with_(name="err_attn_mla", n_req=2),
                               W.MLA_128K.with_(name="err_attn_mla_tc", n_req=2, n_layer=1, ctx0=2048, budget_blocks=256,
                                                cap_blocks=384, n_heavy=20)], ids=["tma", "cp_async", "tcgen05"])
@pytest.mark.parametrize("bad", ["slot_past_end", "slot_negative", "block_past_end", "count"])
def test_attention_refuses_bad_indices(w, bad):
    g = GpuCase(w, [w.ctx0, w.ctx0 - 77])
    n = min(w.budget_blocks, 16)
    sel, nsel = _first_blocks(g, n)
    sos = torch.zeros_like(sel)
    g.ctx.cache_update(0, sel, nsel, g.ctx_len, sos, g.stats)
    q = torch.from_numpy(g.qs.queries(0)[0].view(np.int16)).cuda()
    ref = torch.zeros((w.n_req, w.n_q_head, w.d_v), dtype=torch.float32, device="cuda")
    g.ctx.sparse_decode_attn(0, q, sel, sos, nsel, g.ctx_len, ref)
    torch.cuda.synchronize()
    assert g.ctx.poll_error() == 0
    r, h = 0, w.n_kv_head - 1
    sel_b, sos_b, nsel_b = sel.clone(), sos.clone(), nsel.clone()
    if bad == "slot_past_end":
        sos_b[r, h, 2] = w.cap_blocks
    elif bad == "slot_negative":
        sos_b[r, h, 2] = -3
    elif bad == "block_past_end":
        sel_b[r, h, n - 1] = (w.ctx0 + w.block_size - 1) // w.block_size
    else:
        nsel_b[r, h] = w.budget_blocks + 1
    out = torch.full_like(ref, 7.0)
    g.ctx.sparse_decode_attn(0, q, sel_b, sos_b, nsel_b, g.ctx_len, out)
    torch.cuda.synchronize()
    assert g.ctx.poll_error() == BAD_INDEX
    G = w.group
    heads = slice(h * G, (h + 1) * G)
    keep = torch.ones(w.n_req, w.n_q_head, dtype=torch.bool)
    keep[r, heads] = False
    assert torch.equal(out.cpu()[keep], ref.cpu()[keep])                 # other units untouched
    assert torch.isfinite(out[r, heads]).all()
    g.close()


def test_bind_rejects_unmapped_host_memory():
    w = W.TINY.with_(name="err_bind")
    g = GpuCase(w)
    # pageable memory of the full history size: not registered with the device
    k = np.zeros((w.n_layer, w.n_req, w.n_kv_head, w.max_ctx, w.d_k), np.int16)
    v = np.zeros_like(k)
    import ctypes
    import sparse_kv_cache_decode_gb300 as K
    L = K.lib()
    st = L.kvs_bind_host_kv(g.ctx.h, k.ctypes.data, v.ctypes.data)
    assert st == HOST_MEM
    assert L.kvs_bind_host_kv(g.ctx.h, None, None) == INVALID_ARG
    assert L.kvs_bind_host_kv(g.ctx.h, g.k_host.data_ptr(), None) == INVALID_ARG   # V missing
    g.close()


def test_invalid_arguments_are_refused_before_launch():
    import sparse_kv_cache_decode_gb300 as K
    w = W.TINY_LOOKAHEAD.with_(name="err_args")
    g = GpuCase(w)
    L = K.lib()
    before = g.ctx.launch_count()
    scores = torch.zeros((w.n_req, w.n_kv_head, g.nb_max), dtype=torch.float32, device="cuda")
    q = torch.zeros((w.n_req, w.n_draft, w.n_q_head, w.d_k), dtype=torch.int16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert L.kvs_score_blocks(g.ctx.h, 1, q.data_ptr(), 1, g.index.data_ptr(), g.ctx_len.data_ptr(),
                              scores.data_ptr(), s) == INVALID_ARG                       # layer 1 of 1
    assert L.kvs_score_blocks(g.ctx.h, 0, q.data_ptr(), w.n_draft + 1, g.index.data_ptr(), g.ctx_len.data_ptr(),
                              scores.data_ptr(), s) == INVALID_ARG                       # nq > max_score_q
    assert L.kvs_score_blocks(g.ctx.h, 0, q.data_ptr(), 0, g.index.data_ptr(), g.ctx_len.data_ptr(),
                              scores.data_ptr(), s) == INVALID_ARG
    assert L.kvs_topk_select(g.ctx.h, None, g.ctx_len.data_ptr(), None, None, s) == INVALID_ARG
    assert L.kvs_layer_prefetch(g.ctx.h, 0, None, None, None, None, s) == INVALID_ARG   # no layer below 0
    assert L.kvs_decode_step(g.ctx.h, -1, q.data_ptr(), None, 1, None, None, g.index.data_ptr(),
                             g.ctx_len.data_ptr(), scores.data_ptr(), None, None, None, s, None) == INVALID_ARG
    assert g.ctx.launch_count() == before
    g.close()
