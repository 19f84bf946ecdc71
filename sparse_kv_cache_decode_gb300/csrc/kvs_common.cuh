// Internal declarations shared by the libkvs translation units (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvs.h"

namespace kvs {

// Shape and policy of one context, as the kernels see it (passed by value).
struct Dims {
  int B, NL, Hq, Hkv, G;
  int dk, dv, v_shares_k;
  int bs, max_ctx, nb_max;
  int Kb, n_sink, n_recent, C, max_nq, lookahead, max_prefetch;
  int evict_importance;  // victims least important first (else least recently used)
  int bound;             // blocks summarised by [max | min] keys and scored by the upper bound
  int didx;              // index row width: dk (block-mean key) or 2 * dk ([max | min] summary)
  int fp8;               // history and slot pools hold E4M3 codes (1 byte per element)
  int ebytes;            // bytes per stored K/V element: 2 (bf16) or 1 (E4M3)
  float k_scale, v_scale;
  int U;                 // units per layer = B * Hkv
  float scale;
  unsigned timeout_us;
  int row_bytes;         // host bytes moved per token: ebytes * (dk + (v_shares_k ? 0 : dv))
};

// Device pointers of one layer.
struct Layer {
  int layer;
  __nv_bfloat16* kpool;  // [U][C][bs][dk]
  __nv_bfloat16* vpool;  // [U][C][bs][dv] (nullptr when v_shares_k)
  int* block2slot;       // [U][nb_max]
  int* slot2block;       // [U][C]
  unsigned* stamp;       // [U][C]
  unsigned* clock;       // [U]
  int* pend_sel;         // [U][Kb]  selection the next lookahead attention reads
  int* pend_slot;        // [U][Kb]
  int* pend_n;           // [U]      -1: none yet
  // A lookahead update stages the selection it made here and marks the unit; the fetch that
  // follows it (which runs after the layer's attention over the current pending selection has
  // finished) commits the staged copy to pend_*, so attention and update may run concurrently.
  int* next_sel;         // [U][Kb]
  int* next_slot;        // [U][Kb]
  int* next_n;           // [U]
  int* next_commit;      // [U]      1: next_* awaits its commit
  float* scores;         // [U][nb_max]   scratch
  int* sel;              // [U][Kb]       scratch (fused step)
  int* nsel;             // [U]
  int* slot_of_sel;      // [U][Kb]
  int* fetch_blk;        // [U][C]  blocks to copy host -> slot (misses or prefetches)
  int* fetch_slot;       // [U][C]
  int* n_fetch;          // [U]
  float* attn_part;      // [U][n_split_max][Hq/Hkv][dv] partial outputs
  float* attn_ml;        // [U][n_split_max][Hq/Hkv][2] partial (max, sum)
  unsigned* unit_done;   // [U] CTAs finished per unit in the current attention launch (0 between launches)
  uint8_t* miss_flag;    // [U][Kb] selected position i was a miss in the last update (fetched, not resident)
  unsigned* score_done;  // [U] scoring CTAs finished per unit in the current layer-kernel launch (0 between launches)
  const __nv_bfloat16* host_k;  // device-mapped host history of this layer [B][Hkv][max_ctx][dk]
  const __nv_bfloat16* host_v;  // [B][Hkv][max_ctx][dv] or nullptr
  unsigned* err;         // sticky status word (shared by all layers)
  const CUtensorMap* tmK; // host copies of the 2D tensor maps over the K / V slot pools (or nullptr)
  const CUtensorMap* tmV;
};

constexpr int kAttnSplitMax = 32;

// Programmatic dependent launch.  The step's kernels are launched with programmatic stream
// serialisation (launch_pdl), so a kernel's CTAs may be scheduled while the kernel before it in
// the stream is still running; each such kernel therefore begins with kvs_pdl_entry(): wait until
// the preceding grid has completed and its writes are visible (before any global memory access),
// then allow the next kernel's CTAs to be scheduled.  Without the launch attribute both
// instructions are no-ops.
__device__ __forceinline__ void kvs_pdl_entry() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// launch_pdl with thread-block clusters of cluster_x CTAs along x (grid.x a multiple of it).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                      unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

__device__ __forceinline__ void set_error(unsigned* err, unsigned code) {
  atomicCAS(err, 0u, code);
}

__device__ __forceinline__ int n_blocks_of(int L, int bs) { return (L + bs - 1) / bs; }

// Orderable key of an fp32 score: larger score -> larger key; -0.0 and +0.0 share a key;
// every NaN maps to 0, below -inf (whose key is 0x007FFFFF).
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;      // NaN
  if (u == 0x80000000u) u = 0u;                         // -0.0 -> +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Chunk c (8 bf16 values) of one scoring row as the scoring kernels stage it: the query row
// itself (block-mean index), or [max(q, 0) | min(q, 0)] for the [max | min] summaries, whose dot
// product with the summary row is sum_d max(q_d mx_d, q_d mn_d) (exact: the kept values are q's).
__device__ __forceinline__ uint4 score_row_chunk(const __nv_bfloat16* qrow, int c, const Dims& d) {
  if (!d.bound) return reinterpret_cast<const uint4*>(qrow)[c];
  const int nc = d.dk / 8;
  const bool neg = c >= nc;
  uint4 v = reinterpret_cast<const uint4*>(qrow)[neg ? c - nc : c];
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = w[i] & 0xffffu, hi = w[i] >> 16;
    const float flo = __uint_as_float(lo << 16), fhi = __uint_as_float(hi << 16);
    const bool klo = neg ? flo < 0.f : flo > 0.f, khi = neg ? fhi < 0.f : fhi > 0.f;
    w[i] = (klo ? lo : 0u) | ((khi ? hi : 0u) << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// E4M3 code -> fp32 value (exact): normals (1 + m/8) 2^(e-7), subnormals m 2^-9, S.1111.111 NaN.
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u, s = (c & 0x80u) << 24;
  if (e == 15u && m == 7u) return __uint_as_float(0x7fc00000u | s);
  if (e == 0u) {
    const float v = (float)m * 0.001953125f;                           // exact; m = 0 gives +-0
    return s ? -v : v;
  }
  return __uint_as_float(s | ((e + 120u) << 23) | (m << 20));
}

// Two fp32 values -> two E4M3 codes (round to nearest even, saturating to +-448): lo in bits 0-7.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// -------------------------------------------------------------- launchers (one per kernel TU)
cudaError_t launch_index_build(const Dims& d, const Layer& L, __nv_bfloat16* index, const int* ctx_len,
                               cudaStream_t s);
cudaError_t launch_append(const Dims& d, const Layer& L, const __nv_bfloat16* k_new,
                          const __nv_bfloat16* v_new, __nv_bfloat16* index, const int* ctx_len, cudaStream_t s);
cudaError_t launch_advance(int B, int* ctx_len, cudaStream_t s);
cudaError_t launch_touch_pages(const void* base, size_t bytes, unsigned* sink, cudaStream_t s);
cudaError_t launch_score(const Dims& d, const __nv_bfloat16* index, const __nv_bfloat16* q, int nq,
                         const int* ctx_len, float* scores, unsigned* err, cudaStream_t s);
// Scratch of the two-phase top-K (long contexts): per (unit, chunk) up to K_b kept candidates.
struct TopkScratch {
  uint32_t* key;  // [U][P][Kb]
  int* idx;       // [U][P][Kb]
  int* cnt;       // [U][P]
};
int topk_chunks(const Dims& d);   // P, or 0 when one pass per unit is used
cudaError_t launch_topk(const Dims& d, const float* scores, const int* ctx_len, int* sel, int* nsel,
                        unsigned* err, cudaStream_t s, const TopkScratch* scratch);
cudaError_t launch_cache_update(const Dims& d, const Layer& L, const int* sel, const int* nsel, const int* ctx_len,
                                int* slot_of_sel, const float* scores, kvs_stats* stats, cudaStream_t s);
// Top-K and cache update of each unit in one kernel (contexts of at most 16384 blocks).
int select_update_fusable(const Dims& d);
// Overlapped lookahead layer in one kernel: attention over the pending selection, scoring with the
// drafts, top-K and cache update (GQA groups of up to 8, the TMA attention path, the mma.sync
// scoring path with up to 32 scoring rows, at most one unit per SM).
int layer_kernel_supported(const Dims& d, int nq, bool have_tmaps);
cudaError_t launch_layer(const Dims& d, const Layer& L, const __nv_bfloat16* q, const __nv_bfloat16* index,
                         const __nv_bfloat16* sq, int nq, const int* ctx_len, float* out, int* sel, int* nsel,
                         kvs_stats* stats, cudaStream_t s);
// threads: the CTA size (a multiple of 32, at most 512).
cudaError_t launch_select_update(const Dims& d, const Layer& L, const float* scores, const int* ctx_len, int* sel,
                                 int* nsel, int* slot_of_sel, kvs_stats* stats, cudaStream_t s, int threads = 512);
// Restore a layer's cache state from a snapshot (per-unit refetch list, then the maps).
struct SnapshotPlan {
  size_t b2s, s2b, stamp, clock, pend_sel, pend_slot, pend_n, total;
};
SnapshotPlan snapshot_plan(const Dims& d);
cudaError_t launch_restore(const Dims& d, const Layer& L, const unsigned char* snap, cudaStream_t s);
cudaError_t launch_prefetch(const Dims& d, const Layer& L, const int* hint, const int* hint_n, const int* ctx_len,
                            kvs_stats* stats, cudaStream_t s);
cudaError_t launch_fetch(const Dims& d, const Layer& L, const int* ctx_len, cudaStream_t s);
cudaError_t launch_attention(const Dims& d, const Layer& L, const __nv_bfloat16* q, const int* sel,
                             const int* slot_of_sel, const int* nsel, const int* ctx_len, float* out,
                             cudaStream_t s);
int attention_supported(const Dims& d);
bool make_tmap_2d(CUtensorMap* m, void* base, uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows,
                  int elem_bytes = 2);
int score_tc_supported(const Dims& d, int nq);
cudaError_t launch_score_tc(const Dims& d, const __nv_bfloat16* index, const __nv_bfloat16* q, int nq,
                            const int* ctx_len, float* scores, unsigned* err, cudaStream_t s);
int attention_tma_supported(const Dims& d);
int attention_tma_partials(const Dims& d);
// phase: 0 all selected positions; 1 the positions that hit in the layer's last update, partials
// kept; 2 those that missed, then every partial merged (1 and 2 in that order on one stream).
cudaError_t launch_attention_tma(const Dims& d, const Layer& L, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                 const __nv_bfloat16* q, const int* sel, const int* slot_of_sel, const int* nsel,
                                 const int* ctx_len, float* out, cudaStream_t s, int phase = 0);
int attention_split(const Dims& d, int* n_split, int* blocks_per_split);
// MLA attention on tcgen05 (128 heads sharing 576-dim latent rows, bf16): the split of the unit's
// selection over CTAs, or 0 when the shape is not served.
int attention_mla_tc_split(const Dims& d, int* n_split, int* blocks_per_split);
int attention_mla_tc_supported(const Dims& d);
cudaError_t launch_attention_mla_tc(const Dims& d, const Layer& L, const __nv_bfloat16* q, const int* sel,
                                    const int* slot_of_sel, const int* nsel, const int* ctx_len, float* out,
                                    cudaStream_t s);
int score_supported(const Dims& d);

// Raise `kernel`'s dynamic shared-memory limit to at least `bytes` on the current device.  The
// attribute belongs to the current device's context, so it is tracked per (kernel, device); safe
// to call from several host threads.
cudaError_t set_max_dynamic_smem(const void* kernel, int bytes);
// Streaming multiprocessors of the current device (looked up once per device).
int device_sm_count();

}  // namespace kvs
