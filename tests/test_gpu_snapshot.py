"""Cache snapshot and restore through the C ABI (kvs_cache_snapshot / kvs_cache_restore), for
speculative rollback: the state saved before some steps is put back, and every slot those steps
overwrote is fetched again from the host history.  Checked against the oracle's restore
(oracle.cache.cache_restore): the cache state after the restore, the contents of every resident
slot, and then further steps, which must follow the oracle exactly (integer-valued inputs, so
every score and selection is exact)."""
import numpy as np
import pytest

import workload as W
from kvs_harness import STAT_KEYS, GpuCase, compare_step as _compare_step

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

CASES = [
    (W.TINY.with_(name="snap_sync_int", n_req=2, n_layer=2, int_scale=2.0), [4096, 2999], False),
    (W.TINY_LOOKAHEAD.with_(name="snap_la_int_cs", n_req=2, n_layer=2, int_scale=2.0), [4096, 3100], True),
    (W.TINY.with_(name="snap_imp_int", n_req=2, int_scale=2.0, evict_policy="importance"), [4096, 1500], False),
]


def _check_state_and_slots(g, o):
    w = g.w
    for l in range(w.n_layer):
        b2s, s2b, st, clk = g.ctx.cache_export(l)
        kp, vp = g.ctx.slot_pool_tensors(l)
        kp = kp.cpu().numpy().view(np.uint16)
        vp = None if vp is None else vp.cpu().numpy().view(np.uint16)
        for r in o.reqs:
            for h in range(w.n_kv_head):
                u = r * w.n_kv_head + h
                c = o.cache[(l, r, h)]
                np.testing.assert_array_equal(s2b[u], c.slot2block, err_msg=f"slot2block {(l, r, h)}")
                np.testing.assert_array_equal(b2s[u], c.block2slot, err_msg=f"block2slot {(l, r, h)}")
                np.testing.assert_array_equal(st[u].astype(np.int64), c.stamp, err_msg=f"stamp {(l, r, h)}")
                assert int(clk[u]) == c.clock
                L = o.L[r]
                for s, b in enumerate(c.slot2block):
                    if b < 0:
                        continue
                    rows = min(w.block_size, L - b * w.block_size)
                    t0 = b * w.block_size
                    np.testing.assert_array_equal(kp[u, s, :rows], g.k_np[l, r, h, t0:t0 + rows],
                                                  err_msg=f"K slot {(l, r, h)} {s}")
                    if vp is not None:
                        np.testing.assert_array_equal(vp[u, s, :rows], g.v_np[l, r, h, t0:t0 + rows])


@pytest.mark.parametrize("w,lens,copy_stream", CASES, ids=[c[0].name for c in CASES])
def test_restore_puts_state_and_slots_back(w, lens, copy_stream):
    g = GpuCase(w, lens, copy_stream=copy_stream)
    o = g.oracle()
    cum = {l: {k: 0 for k in STAT_KEYS} for l in range(w.n_layer)}

    def step(t):
        q, d, nk, nv = g.step_inputs(t)
        g.gpu_step(q, d, nk, nv)
        out_ref, recs = o.step(q, d, nk, nv)
        _compare_step(g, o, out_ref, recs, cum, exact=True)

    for t in range(3):
        step(t)
    nbytes = g.ctx.snapshot_bytes()
    snaps = [torch.empty(nbytes + 256, dtype=torch.uint8, device="cuda") for _ in range(w.n_layer)]
    views = [sb[(256 - sb.data_ptr() % 256) % 256:][:nbytes] for sb in snaps]
    for l in range(w.n_layer):
        g.ctx.cache_snapshot(l, views[l])
    o_snap = o.snapshot()
    torch.cuda.synchronize()
    for t in range(3, 7):                 # the steps that are rolled back
        step(t)
    stats_before = g.stats.cpu().numpy().copy()
    for l in range(w.n_layer):
        g.ctx.cache_restore(l, views[l], g.ctx_len)
    o.restore(o_snap)
    torch.cuda.synchronize()
    assert g.ctx.poll_error() == 0
    np.testing.assert_array_equal(g.stats.cpu().numpy(), stats_before)   # restores do not count
    _check_state_and_slots(g, o)
    for t in range(7, 11):                # and the steps after the rollback follow the oracle
        step(t)
    assert g.ctx.poll_error() == 0


def test_snapshot_rejects_misaligned_buffer():
    import sparse_kv_cache_decode_gb300 as K
    w = W.TINY.with_(name="snap_args")
    g = GpuCase(w)
    buf = torch.empty(g.ctx.snapshot_bytes() + 512, dtype=torch.uint8, device="cuda")
    base = (256 - buf.data_ptr() % 256) % 256
    with pytest.raises(K.KvsError) as e:
        g.ctx.cache_snapshot(0, buf.data_ptr() + base + 4)
    assert e.value.status == 1
    assert g.ctx.snapshot_bytes() > 0
