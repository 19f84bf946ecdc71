/*
 * kvs.h -- C ABI of libkvs: one decode step of top-K sparse KV-cache attention with the
 * full KV history in pinned host memory and a fixed-size GPU working-set cache (sm_103a).
 *
 * Method sources (page title, section):
 *  [SPEC]  "KV Cache 塞不进 HBM 了：投机式稀疏预取如何把长上下文推理再提速 2-25 倍" (tuntang.top):
 *          2.1 SpeContext (head-level selection; elastic loading to_load = S_now - S_last on
 *          another CUDA stream), 2.3 SparseSpec-L (sink + recent + top tokens), 3 step 1
 *          (per-step select -> delta -> async prefetch -> attention), 3 step 3 (GQA: element-wise
 *          max of scores within a group, then top-K per group; MLA: select on the latent cache).
 *  [OASIS] "OasisKV: 利用 Lookahead 稀疏预取将解码 KV 缓存扩展到 HBM 之外" (ai-feeds.com), 方法:
 *          key module 1 (exact foreground attention over the sparse HBM KV), 2 (lookahead drafts
 *          score KV blocks), 3 (delta selection and a capped HBM cache).
 *  [HISP]  "长上下文 LLM 为何总被显存"卡脖子"？" (HiSparse, papers.ananclaw.com): insight 1 (full KV
 *          in host memory, fixed-size GPU cache, exact outputs, indexer-agnostic), insight 2
 *          (fused hit detection + LRU replacement + host-to-device fetch inside the decode CUDA
 *          graph, no host sync, atomic in-kernel LRU), insight 3 (cross-layer prefetch).
 *  [KVC]   "当上下文冲破百万：KV-Cache压缩技术的工程原理与2026年工业实践" (jiusizaji.com), 1.1 (KV
 *          size), 2.2 GQA, 2.3 MLA.
 *
 * Terms.  B requests, N_l layers, H_q / H_kv query / kv heads (G = H_q / H_kv; q head h uses kv
 * head h / G), d_k / d_v head dims, bs tokens per block, K_b blocks per selection, C cache slots
 * per unit.  A unit is one (request, layer, kv-head); a layer's units are numbered
 * u = request * H_kv + kv_head.  ctx_len[r] = L_r tokens present for request r; n_b(L) = ceil(L/bs).
 *
 * Layouts (row-major, bf16 = 16-bit patterns; history and slot pools in E4M3 bytes when
 * kv_dtype is FP8):
 *   host K      [N_l][B][H_kv][max_ctx][d_k]      pinned, device-mapped (see kvs_bind_host_kv)
 *   host V      [N_l][B][H_kv][max_ctx][d_v]      absent when v_shares_k (V = first d_v of K row)
 *   index       [N_l][B][H_kv][n_b(max_ctx)][d_idx] device; block summaries (kvs_index_build):
 *                                                 d_idx = d_k (mean key) or 2 d_k ([max | min])
 *   q           [B][H_q][d_k]                     one layer's attention queries
 *   score_q     [B][nq][H_q][d_k]                 one layer's scoring queries (drafts)
 *   scores      [B][H_kv][n_b(max_ctx)] fp32      one layer's block scores
 *   sel         [B][H_kv][K_b] int32              selected block ids, ascending; nsel [B][H_kv]
 *   slot_of_sel [B][H_kv][K_b] int32              cache slot of each selected block
 *   out         [B][H_q][d_v] fp32                one layer's attention output
 *   k_new/v_new [B][H_kv][d_k] / [d_v] bf16       one layer's appended token (16-byte aligned)
 *   ctx_len     [B] int32 (device)
 *
 * Ownership.  The caller owns every buffer.  The device workspace (kvs_workspace_bytes) holds
 * the slot pools, the per-unit cache state, per-layer scratch and the error word; the library
 * carves it and never allocates device memory.  The pinned host history is registered by the
 * caller (cudaHostAlloc / cudaHostRegister with the mapped flag) and never freed here.
 *
 * Calls.  Every compute call is asynchronous on the given stream, performs no host sync and
 * is capturable in a CUDA graph (exceptions: kvs_create, kvs_bind_host_kv, kvs_cache_export,
 * kvs_poll_error, kvs_destroy).  The return value reports argument and launch errors only.
 * Errors found on the device (capacity overflow, bad block id, a wait that ran out of time)
 * set a sticky status word that kvs_poll_error reads after the caller synchronises; no
 * kernel traps.  Calls on the same layer must not overlap on the GPU.  The workspace holds two
 * copies of the block-score and top-K candidate scratch, one per layer parity: kvs_decode_step
 * calls on layers of the same parity must not overlap (kvs_decode_step orders its own selection
 * chains so), and a kvs_topk_select call (which uses the even copy) must not overlap an even
 * layer's step; kvs_layer_prefetch may run beside them.
 */
#ifndef KVS_H_
#define KVS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kvs_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  KVS_OK = 0,
  KVS_ERR_INVALID_ARG = 1,   /* a pointer, size or config value is out of range */
  KVS_ERR_CUDA = 2,          /* a CUDA runtime call or launch failed */
  KVS_ERR_CAPACITY = 3,      /* a cache had fewer victim slots than misses */
  KVS_ERR_TIMEOUT = 4,       /* a device wait ran out of time */
  KVS_ERR_HOST_MEM = 5,      /* host history not pinned/mapped, or not bound */
  KVS_ERR_NOT_SUPPORTED = 6, /* a shape this build has no kernel for */
  KVS_ERR_BAD_INDEX = 7      /* the device saw a block id outside [0, n_b(L)) */
} kvs_status;

typedef struct {
  int n_req, n_layer, n_q_head, n_kv_head;
  int d_k, d_v;        /* multiples of 8; d_v <= d_k when v_shares_k */
  int v_shares_k;      /* 1: MLA latent row; V is the first d_v entries of the K row [KVC 2.3] */
  int block_size;      /* bs >= 1 */
  int max_ctx;         /* tokens per unit in the host history (capacity, including appends) */
  int budget_blocks;   /* K_b */
  int n_sink, n_recent;/* forced blocks at the start / end of the context [SPEC 2.3] */
  int cap_blocks;      /* C >= K_b cache slots per unit [OASIS module 3] */
  int max_score_q;     /* largest nq passed to score calls (1 in sync mode) */
  int lookahead;       /* 1: attention uses the selection made by the previous step [SPEC 3.1] */
  int max_prefetch;    /* per-unit cap of kvs_layer_prefetch; 0 -> C - K_b */
  float softmax_scale; /* 0 -> 1/sqrt(d_k) rounded to fp32 */
  unsigned wait_timeout_us; /* bound on device waits (0 -> 2000000 us) */
  int evict_policy;    /* KVS_EVICT_LRU (0) or KVS_EVICT_IMPORTANCE (1) [OASIS module 3, HISP insight 2] */
  int score_mode;      /* KVS_SCORE_MEAN (0) or KVS_SCORE_BOUND (1): how blocks are summarised and scored */
  int kv_dtype;        /* KVS_KV_BF16 (0) or KVS_KV_FP8_E4M3 (1): the history's and the slot pools' format */
  float k_scale, v_scale; /* E4M3: a stored key is decode(code) * k_scale, a value decode(code) * v_scale (0 -> 1) */
} kvs_config;

/* KV storage format [KVC 3.2: FP8 E4M3 keeps accuracy at half the bytes].  BF16: host history and
 * slot pools hold bf16.  FP8_E4M3: they hold E4M3 codes (bias 7, 3 mantissa bits, largest finite
 * 448, no infinity) of value / scale; host K/V rows are d_k / d_v bytes.  Index keys (bf16) are
 * built from the fp32 values fp32(decode(code) * k_scale); attention computes the logits as
 * (softmax_scale * k_scale) * (q . decode(code_k)) and the output as v_scale * sum p decode(code_v)
 * / sum p, with every code widened exactly to bf16 for the tensor-core tiles; appended bf16 tokens
 * are quantised on arrival (round to nearest even, saturating to +-448).  Supported with block-mean
 * scoring, separate K and V of head dim 128 and block sizes that are multiples of 16. */
enum { KVS_KV_BF16 = 0, KVS_KV_FP8_E4M3 = 1 };

/* Block summaries and scores.  MEAN: the index row of a block is its mean key (d_idx = d_k) and
 * the score is the mean token logit q . ik.  BOUND: the index row is [max | min] of its present
 * keys per dimension (d_idx = 2 d_k, exact bf16) and the score is the query-aware upper bound
 * sum_d max(q_d max_d, q_d min_d) of the block's largest token logit (the Quest rule; the pages
 * name Quest among the selector families the host-KV cache serves [HISP insight 1]). */
enum { KVS_SCORE_MEAN = 0, KVS_SCORE_BOUND = 1 };

/* Victim order of the cache update.  LRU: least recently used first, by (stamp, slot).
 * IMPORTANCE: least important first: the block's score in the scoring that made the selection
 * (NaN lowest, -0.0 == +0.0), ties by slot.  Both take empty slots first; the cross-layer
 * prefetch always picks its victims by LRU (no scores of the destination layer exist yet). */
enum { KVS_EVICT_LRU = 0, KVS_EVICT_IMPORTANCE = 1 };

/* Per-layer counters, accumulated with atomics into a caller buffer kvs_stats[N_l]. */
typedef struct {
  unsigned long long hits, misses, evictions, prefetched, prefetch_hits, pin_fallbacks;
  unsigned long long bytes_fetched; /* host -> device bytes of misses and prefetches */
} kvs_stats;

typedef struct kvs_ctx kvs_ctx;

/* Device bytes the workspace of `cfg` needs (0 when cfg is invalid). */
size_t kvs_workspace_bytes(const kvs_config* cfg);

/* Validate cfg and carve d_workspace (>= kvs_workspace_bytes, 256-byte aligned device memory).
 * Clears the cache state (all slots empty and zero-filled, clocks 0) on the current device,
 * synchronously.
 * Errors: KVS_ERR_INVALID_ARG (bad cfg, short or misaligned workspace), KVS_ERR_CUDA. */
kvs_status kvs_create(const kvs_config* cfg, void* d_workspace, size_t workspace_bytes, kvs_ctx** out);
kvs_status kvs_destroy(kvs_ctx* ctx);

/* Bind the pinned host history [HISP insight 1]: h_k, h_v in the layouts above (h_v NULL when
 * v_shares_k).  The memory must be page-locked and mapped into the device address space.  The
 * device reads one word of every 4 KiB page once (synchronously), so the translations of the
 * whole history exist before the first fetch.  Errors: KVS_ERR_HOST_MEM when a pointer is not
 * page-locked host memory mapped into the device address space (pageable memory is refused even
 * where the device could reach it). */
kvs_status kvs_bind_host_kv(kvs_ctx* ctx, void* h_k, void* h_v);

/* Build the block summaries of one layer from the host history (setup after prefill).  MEAN:
 * ik[b] = bf16_rne( (sum over present tokens t of block b, ascending, of fp32 k_t) / n_b ); reading
 * of [OASIS module 2] "per-block importance": by linearity q.ik[b] is the block's mean token logit.
 * BOUND: ik[b] = [max_t k_t | min_t k_t] per dimension over the present tokens (ties keep the
 * earliest token's value).  Blocks >= n_b(ctx_len[r]) are left untouched. */
kvs_status kvs_index_build(kvs_ctx* ctx, int layer, void* d_index, const int* d_ctx_len, kvs_stream_t stream);

/* Block scores of one layer [SPEC 3 step 3, OASIS module 2]:
 * s[r][h][b] = scale * max over j < nq and q heads g of group h of (score_q[r][j][g] . ik[b])
 * (BOUND: of sum_d max(q_d max_d, q_d min_d), evaluated as [max(q,0) | min(q,0)] . ik[b]),
 * fp32 with fp32 accumulation of exact bf16 products, for b < n_b(ctx_len[r]); other entries
 * are left untouched.  nq in [1, max_score_q].  Kernels: tcgen05 tensor cores for 64-256 scoring
 * rows per unit (nq * G) with d_k a multiple of 64; mma.sync tiles for up to 128 rows with d_k 128
 * or 576.  A configuration any of whose call widths 1..max_score_q has neither is refused with
 * KVS_ERR_NOT_SUPPORTED. */
kvs_status kvs_score_blocks(kvs_ctx* ctx, int layer, const void* d_score_q, int nq, const void* d_index,
                            const int* d_ctx_len, float* d_scores, kvs_stream_t stream);

/* Selection [SPEC 2.3, 3 step 1]: with nb = n_b(ctx_len[r]), all blocks when nb <= K_b; else the
 * sink blocks [0, n_sink), the recent blocks [nb - n_recent, nb) and the top K_b - |forced| other
 * blocks by (score desc, block asc), NaN below -inf, -0.0 == +0.0.  Output ascending in
 * sel[r][h][0 .. nsel-1]; nsel = min(K_b, nb).  When n_b(max_ctx) exceeds 16384 blocks the
 * selection runs in two phases over chunks of 16384 blocks (same result). */
kvs_status kvs_topk_select(kvs_ctx* ctx, const float* d_scores, const int* d_ctx_len, int* d_sel, int* d_nsel,
                           kvs_stream_t stream);

/* Cache update of one layer [SPEC 2.1, OASIS module 3, HISP insight 2], then the fetch of the
 * misses from host memory into their slots (rows < L of each block), on `stream`:
 *   clock += 1; hits = selected blocks already resident; misses = the delta (ascending);
 *   victims = slots that are empty or hold a block neither selected nor pinned, in the order of
 *   cfg.evict_policy (least recently used by (stamp, slot), or least important by d_scores);
 *   miss i takes victim i; every selected block is stamped 2*clock.
 * In lookahead mode the blocks of the layer's previous selection are pinned (they are what the
 * pending attention reads); with too few victims the pins are dropped (pin_fallbacks).  Writes
 * slot_of_sel; adds to d_stats[layer] when d_stats is not NULL.  d_scores [B][H_kv][n_b(max_ctx)]
 * fp32: the block scores behind d_sel, required under KVS_EVICT_IMPORTANCE (else unused, may be
 * NULL).  Device errors: KVS_ERR_CAPACITY when even without pins the victims are fewer than the
 * misses; KVS_ERR_BAD_INDEX for a block id out of range or a selection that is not strictly
 * ascending (the unit's state is then left unchanged). */
kvs_status kvs_cache_update(kvs_ctx* ctx, int layer, const int* d_sel, const int* d_nsel, const int* d_ctx_len,
                            int* d_slot_of_sel, const float* d_scores, kvs_stats* d_stats, kvs_stream_t stream);

/* Speculative rollback of a layer's cache state [KVC 6.1: save the block table before the drafts,
 * copy it back when they are rejected].  The snapshot holds the maps, stamps, clocks and the
 * pending lookahead selection of every unit of the layer, in a caller device buffer of
 * kvs_snapshot_bytes(cfg) bytes (256-byte aligned).  kvs_cache_snapshot copies them there with
 * device-to-device copies on `stream`.  kvs_cache_restore copies them back and, because evicted
 * slots of this cache are overwritten, fetches again from the host history every slot whose block
 * differs from the snapshot's (when the snapshot's slot held a block; rows < ctx_len), so that
 * state and slot contents are exactly as at the snapshot.  Both are asynchronous and capturable;
 * the caller orders them after the layer's pending fetches (kvs_join) and restores ctx_len itself.
 * Restores do not add to the counters. */
size_t kvs_snapshot_bytes(const kvs_config* cfg);
kvs_status kvs_cache_snapshot(kvs_ctx* ctx, int layer, void* d_snapshot, kvs_stream_t stream);
kvs_status kvs_cache_restore(kvs_ctx* ctx, int layer, const void* d_snapshot, const int* d_ctx_len,
                             kvs_stream_t stream);

/* Exact decode attention over the selected slots [OASIS module 1, HISP insight 1]:
 * out[r][g] = sum_t softmax_t(scale * q[r][g] . k_t) v_t over the tokens t < ctx_len[r] of the
 * blocks sel[r][h] (h = g / G), read from their slots; fp32 accumulation, fp32 output.
 * Shapes: d_k = d_v = 128 with G <= 16 (TMA-fed kernel when block_size is a multiple of 16), or
 * MLA (v_shares_k, d_k 576, d_v <= 512, a multiple of 128) with G <= 16, G = 128, or (d_v = 512)
 * G = 32, 64 or 96.  bf16 MLA with G = 128 and d_v = 512 runs on the tensor cores (tcgen05: S, O
 * and P in tensor memory); the other MLA shapes on mma.sync tiles.  Others KVS_ERR_NOT_SUPPORTED. */
kvs_status kvs_sparse_decode_attn(kvs_ctx* ctx, int layer, const void* d_q, const int* d_sel,
                                  const int* d_slot_of_sel, const int* d_nsel, const int* d_ctx_len,
                                  float* d_out, kvs_stream_t stream);

/* The fused decode step of one layer [SPEC 3 step 1, HISP insight 2]:
 *   sync mode:      [append] -> score(score_q or q) -> select -> update + fetch -> attention
 *   lookahead mode: [append] -> attention over the previous selection, and score(drafts) ->
 *                   select -> update with that selection pinned -> fetch on copy_stream.
 * The first lookahead step of a layer has no previous selection and runs the sync part first.
 * Lookahead with a separate copy_stream overlaps the two halves [SPEC 1, OASIS module 2].  For
 * GQA groups of up to 8 heads on the TMA attention path, with up to 32 scoring rows, one kernel on
 * `stream` runs both on a fixed split of the SMs: attention CTAs, scoring CTAs, and per unit the
 * last scoring CTA to finish runs the select + update; the fetch on copy_stream follows it.
 * Otherwise the selection chain (score, select, update) runs on one of two streams the context
 * owns (one per layer parity), starting once the work enqueued on `stream` before this call (the
 * layer below's attention) has finished, beside this layer's attention on `stream` and the chain
 * of the layer below; the fetch on copy_stream waits for the chain and the attention.
 * k_new / v_new NULL: no append (else as kvs_append, after kvs_advance_ctx).  d_score_q NULL
 * scores with d_q (nq = 1).  copy_stream NULL or == stream: the fetch runs on stream.  With a
 * separate copy_stream the caller calls kvs_join before reusing the layer or ending a capture.
 * d_sel_out / d_nsel_out (optional) receive the selection made in this call. */
kvs_status kvs_decode_step(kvs_ctx* ctx, int layer, const void* d_q, const void* d_score_q, int nq,
                           const void* d_k_new, const void* d_v_new, void* d_index, const int* d_ctx_len,
                           float* d_out, kvs_stats* d_stats, int* d_sel_out, int* d_nsel_out,
                           kvs_stream_t stream, kvs_stream_t copy_stream);

/* Make `stream` wait for every fetch issued on copy streams by kvs_decode_step and every
 * kvs_layer_prefetch not yet consumed by an update. */
kvs_status kvs_join(kvs_ctx* ctx, kvs_stream_t stream);

/* Cross-layer prefetch [HISP insight 3] into dst_layer (>= 1) with the hint sel/nsel of the layer
 * below: for each hint block, ascending, not resident, at most max_prefetch per unit: the victim
 * is the least recently used slot that is empty or (stamp < 2*clock and holds no hint block);
 * it is mapped, fetched from host and stamped 2*clock + 1.  Call it before dst_layer's update
 * of the same step; it may run on another stream: it waits for the top-K of the layer below made
 * by kvs_decode_step, and kvs_decode_step(dst_layer) waits for it before its update.
 * It pays only where the layer below's selection foretells this layer's new blocks [HISP insight
 * 3: enable it for selectors that share choices across layers, off otherwise].  Hint blocks this
 * layer never selects are not resident, so they are fetched again at every step, into slots the
 * previous step left unused, which are the ones that give hits when a selection drifts back: the
 * device counters prefetched / prefetch_hits show which case a workload is in, and a smaller
 * max_prefetch bounds the cost. */
kvs_status kvs_layer_prefetch(kvs_ctx* ctx, int dst_layer, const int* d_hint_sel, const int* d_hint_nsel,
                              const int* d_ctx_len, kvs_stats* d_stats, kvs_stream_t stream);

/* ctx_len[r] += 1 for every request (the start of a decode step that appends a token). */
kvs_status kvs_advance_ctx(kvs_ctx* ctx, int* d_ctx_len, kvs_stream_t stream);

/* Append one token per (request, kv-head) to one layer (after kvs_advance_ctx): write it at
 * position ctx_len[r] - 1 of the host history, into the slot of its block when that block is
 * resident, and recompute the block's index key from its present tokens (rule of
 * kvs_index_build).  The KV cache grows by one token per decode step [SPEC introduction]. */
kvs_status kvs_append(kvs_ctx* ctx, int layer, const void* d_k_new, const void* d_v_new, void* d_index,
                      const int* d_ctx_len, kvs_stream_t stream);

/* Copy one layer's cache state to host buffers (synchronous: it waits for all work on the
 * device, because the context's kernels may be on any of the caller's streams; a diagnostic, not
 * for the inside of a pipelined step loop): block2slot [B*H_kv][n_b(max_ctx)],
 * slot2block [B*H_kv][C], stamp [B*H_kv][C], clock [B*H_kv]; any pointer may be NULL. */
kvs_status kvs_cache_export(kvs_ctx* ctx, int layer, int* h_block2slot, int* h_slot2block, unsigned* h_stamp,
                            unsigned* h_clock);

/* Device address of one layer's K and V slot pools, [B*H_kv][C][bs][d_k] and [..][d_v]
 * (V NULL when v_shares_k), for inspection. */
kvs_status kvs_slot_pools(kvs_ctx* ctx, int layer, void** d_k_pool, void** d_v_pool);

/* Read and clear the sticky device status word (synchronous: it waits for all work on the device,
 * as the context's kernels may be on any of the caller's streams; poll between steps).
 * *device_status = KVS_OK when no device-side error happened since the last poll. */
kvs_status kvs_poll_error(kvs_ctx* ctx, kvs_status* device_status);

/* Kernel timers (diagnostics).  After kvs_kernel_timer_arm(ctx, kernel, capacity), the next
 * `capacity` launches of that kernel (by any call, eager or captured in a CUDA graph) are each
 * bracketed by a pair of CUDA events recorded on the launch stream; several kernels can be armed
 * at once.  kvs_kernel_timer_read (synchronous) returns that kernel's summed elapsed milliseconds
 * and number of timed launches.  kernel: one of kvs_kernel_id; capacity 0 disarms it.  Inside
 * kvs_decode_step, when a unit's block scores fit one CTA's shared memory (at most 16384 blocks),
 * top-K and the cache update run as one kernel, timed as KVS_K_UPDATE (KVS_K_TOPK then counts
 * only kvs_topk_select calls and the two-kernel path). */
typedef enum {
  KVS_K_SCORE = 1, KVS_K_TOPK = 2, KVS_K_UPDATE = 3, KVS_K_FETCH = 4, KVS_K_ATTN = 5,
  KVS_K_PREFETCH = 6, KVS_K_APPEND = 7, KVS_K_INDEX = 8
} kvs_kernel_id;
kvs_status kvs_kernel_timer_arm(kvs_ctx* ctx, int kernel, int capacity);
kvs_status kvs_kernel_timer_read(kvs_ctx* ctx, int kernel, double* total_ms, int* n_timed);

/* Number of kernels this context has launched (or captured into graphs) so far. */
unsigned long long kvs_launch_count(kvs_ctx* ctx);

/* Host-link read probe (diagnostics; no counterpart in the pages): n_ctas CTAs of `threads`
 * threads read n_items items of item_bytes each from page-locked, device-mapped host memory at
 * h_base + d_offsets[i] (device array, bytes), with the block fetch's access pattern (one item per
 * warp, 16-byte loads, up to 16 per lane in flight), and write nothing but a sentinel hit count to
 * d_sink[0]; items outside [0, region_bytes) or not 16-byte aligned are skipped and counted in
 * d_sink[1] (the caller zeroes both words).  Timing the call gives the link's SM zero-copy read
 * rate for that pattern.  item_bytes a positive multiple of 16; threads a multiple of 32 in
 * [32, 1024].  Errors: KVS_ERR_INVALID_ARG, KVS_ERR_HOST_MEM (h_base not device-mapped). */
kvs_status kvs_probe_host_read(const void* h_base, size_t region_bytes, const long long* d_offsets, int n_items,
                               int item_bytes, int n_ctas, int threads, unsigned* d_sink, kvs_stream_t stream);

/* Block selection that allocates nothing (no counterpart in the pages: an interface for callers
 * that cannot allocate device memory, e.g. code running inside an allocator hook, or a plug-in in
 * a process whose device memory another runtime owns).  It makes CUDA API calls (device query,
 * symbol lookup, kernel launches), so it must not be called from a stream callback or a
 * cudaLaunchHostFunc host function.  Scores and
 * selects one layer's blocks exactly as kvs_score_blocks followed by kvs_topk_select, without a
 * kvs_ctx or workspace: the block scores live in a file-scope device array of
 * KVS_NOALLOC_MAX_SCORES floats (8 MiB) that every GPU loading the library holds until exit.
 *   cfg          shape and selection policy (validated like kvs_create)
 *   d_score_q    [B][nq][H_q][d_k] bf16 scoring queries, 1 <= nq <= cfg->max_score_q
 *   d_index_layer one layer's index keys [B][H_kv][n_b(max_ctx)][d_k] bf16
 *   d_ctx_len    [B] int32;  d_sel [B][H_kv][K_b] int32 and d_nsel [B][H_kv] int32 outputs
 *   d_status     optional device word that receives device-side errors (sticky), such as
 *                KVS_ERR_BAD_INDEX for a ctx_len above max_ctx.  With d_status NULL such errors
 *                go to a word of the library's own that the caller cannot read, and the units
 *                they hit leave sel / nsel unwritten (stale values from earlier calls): pass a
 *                status word wherever ctx_len is not known to be valid.
 * Returns KVS_ERR_CAPACITY when B * H_kv * n_b(max_ctx) > KVS_NOALLOC_MAX_SCORES (checked before
 * any pointer), KVS_ERR_INVALID_ARG for a bad config, pointer or nq.  The first
 * call on a device looks up the array's device address (cudaGetSymbolAddress); make that first
 * call before any stream capture.  All calls share the array, so calls that overlap on the GPU
 * (other streams, other threads) race; every score a call reads is written by that same call. */
#define KVS_NOALLOC_MAX_SCORES (1 << 21)
kvs_status kvs_select_blocks_noalloc(const kvs_config* cfg, const void* d_score_q, int nq,
                                     const void* d_index_layer, const int* d_ctx_len, int* d_sel, int* d_nsel,
                                     unsigned* d_status, kvs_stream_t stream);

/* E4M3 codes of n bf16 values (device buffers): code[i] = encode(fp32(src[i]) / scale), rounding to
 * nearest even and saturating to +-448 (no counterpart in the pages beyond the format: the
 * quantiser of an FP8 history, the rule the append applies to new tokens).  scale > 0.
 * Errors: KVS_ERR_INVALID_ARG. */
kvs_status kvs_quantize_e4m3(const void* d_src_bf16, void* d_dst, size_t n, float scale, kvs_stream_t stream);

/* Library version string. */
const char* kvs_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KVS_H_ */
