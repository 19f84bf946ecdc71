"""CPU oracle for the sparse KV-cache decode step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg (and its
``--impl reference`` arm) may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls anything here, and this package imports
nothing from the product path.  The two share no code; only the seeded input generator in
``workload/`` feeds both.

What it computes, written plainly (numpy, fp64 where the arithmetic is floating point):

  kv_size      KV-cache size formula 2*L*N_layer*N_kv_head*D_head*P
               ("当上下文冲破百万" KV-cache overview, section 1.1).
  bf16         bf16 round-to-nearest-even from the IEEE-754 definitions.
  index_keys   per-block mean key used to score blocks (a reading: the pages name "attention
               scoring -> per-block importance" without the block summary).
  bound        per-block [max | min] key summaries and the query-aware upper-bound block score
               (second scoring mode; the Quest rule the pages name among selector families).
  scores       block score = scale * max over GQA group heads and scoring queries of q.ik
               (tuntang.top survey, section 3 step 3: element-wise max within a GQA group;
               OasisKV page, key module 2: lookahead drafts score KV blocks).
  select       sink + recent + top-K by (score desc, block asc) (tuntang.top survey, section
               2.3 SparseSpec-L; section 3 step 1 "topk(k=kv_budget)").
  cache        hit detection, delta to_load = S_now - resident, LRU (or least-important)
               victims under a capacity cap, slot assignment, stamps (tuntang.top survey,
               section 2.1 elastic loading; OasisKV page, key module 3; HiSparse page, insights
               1 and 2), the cross-layer prefetch (HiSparse page, insight 3), and snapshot /
               restore for speculative rollback (KV-cache overview, section 6.1).
  attention    exact softmax attention over the selected tokens (OasisKV page, key module 1;
               HiSparse page, insight 1: outputs identical to full KV in HBM).
  step         one decode step over all layers: append, score, select, update, prefetch,
               attend -- sync mode and lookahead-draft mode.

Every function is pinned by tests under ``tests/`` against closed forms, hand-worked
fixtures (``tests/golden/``), brute force or a library routine; see each module's header.
"""
from .bf16 import bf16_to_f32, bf16_to_f64, f32_to_bf16_rne
from .kv_size import kv_cache_bytes, kv_cache_bytes_variant
from .index_keys import index_keys, index_key_block
from .bound import block_scores_bound, index_minmax, index_minmax_block
from .scores import block_scores
from .select import forced_blocks, select_blocks
from .cache import (UnitCache, UpdateResult, PrefetchResult, cache_restore, cache_update, importance_key,
                    layer_prefetch)
from .attention import attend
from .step import OracleDecoder, UnitRecord

__all__ = [
    "bf16_to_f32", "bf16_to_f64", "f32_to_bf16_rne", "kv_cache_bytes", "kv_cache_bytes_variant",
    "index_keys", "index_key_block", "index_minmax", "index_minmax_block", "block_scores", "block_scores_bound", "forced_blocks", "select_blocks", "UnitCache",
    "UpdateResult", "PrefetchResult", "cache_update", "cache_restore", "importance_key", "layer_prefetch", "attend", "OracleDecoder",
    "UnitRecord",
]
