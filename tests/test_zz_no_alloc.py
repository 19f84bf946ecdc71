"""kvs_select_blocks_noalloc: the block-selection entry point for callers that cannot allocate
device memory (for example code running inside an allocator hook, or a plug-in whose process
budgets all device memory elsewhere).  It keeps its block scores in a fixed device array inside
the library instead of a caller workspace.

Checked through the C ABI against the existing entry points (kvs_score_blocks followed by
kvs_topk_select) on the same inputs, on two calls in a row with different queries, so the
second call also shows that scores left in the shared array by the first do not leak in.
Selections are integer results of the same kernels: they must match exactly."""
import numpy as np
import pytest

import workload as W
from kvs_harness import GpuCase

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.mark.parametrize("w,lens", [
    (W.TINY.with_(name="noalloc_tiny", n_req=3), [4096, 1000, 17]),
    (W.TINY_LOOKAHEAD.with_(name="noalloc_drafts", n_req=2), [4096, 2222]),
    # token-level MLA shape above 16384 blocks: tensor-core scoring, and a single-pass top-K over
    # global memory here against the two-phase top-K of the context path
    (W.MLA_128K.with_(name="noalloc_mla_64k", n_req=2, n_layer=1, ctx0=65536, layer_prefetch=False),
     [65536, 65536 - 123]),
])
def test_noalloc_selection_matches_existing_entry_points(w, lens):
    import sparse_kv_cache_decode_gb300 as K
    g = GpuCase(w, lens)
    B, Hkv, Kb = w.n_req, w.n_kv_head, w.budget_blocks
    scores = torch.zeros((B, Hkv, g.nb_max), dtype=torch.float32, device="cuda")
    ref_sel = torch.zeros((B, Hkv, Kb), dtype=torch.int32, device="cuda")
    ref_n = torch.zeros((B, Hkv), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t in range(2):
        q, d, _, _ = g.step_inputs(t)
        rows = torch.from_numpy((d if d is not None else q)[0].view(np.int16)).cuda()
        nq = w.n_score_q
        g.ctx.score_blocks(0, rows, nq, g.index, g.ctx_len, scores)
        g.ctx.topk_select(scores, g.ctx_len, ref_sel, ref_n)
        sel = torch.full((B, Hkv, Kb), -5, dtype=torch.int32, device="cuda")
        nsel = torch.full((B, Hkv), -5, dtype=torch.int32, device="cuda")
        K.select_blocks_noalloc(g.cfg, rows, nq, g.index[0], g.ctx_len, sel, nsel, status)
        torch.cuda.synchronize()
        rn, gn = ref_n.cpu().numpy(), nsel.cpu().numpy()
        np.testing.assert_array_equal(gn, rn)
        rs, gs = ref_sel.cpu().numpy(), sel.cpu().numpy()
        for r in range(B):
            for h in range(Hkv):
                np.testing.assert_array_equal(gs[r, h, :rn[r, h]], rs[r, h, :rn[r, h]], err_msg=f"call {t} unit {(r, h)}")
    assert int(status.item()) == 0
    assert g.ctx.poll_error() == 0


def test_noalloc_rejects_oversized_shapes():
    """The size limit is checked before anything else: with every device pointer NULL the call
    still answers KVS_ERR_CAPACITY (no kernel can be launched on a refused shape)."""
    import sparse_kv_cache_decode_gb300 as K
    w = W.MLA_128K.with_(n_req=32)            # 32 x 131072 block scores > the array's 2^21
    cfg = K.make_config(w)
    with pytest.raises(K.KvsError) as e:
        K.select_blocks_noalloc(cfg, None, 1, None, None, None, None)
    assert e.value.status == 3
