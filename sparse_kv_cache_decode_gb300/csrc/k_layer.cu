// One kernel per layer for the overlapped lookahead step: attention over the pending selection S_t,
// scoring of the layer's blocks with the lookahead drafts, and the selection of S_{t+1} with its
// cache update, on a fixed partition of the CTAs of one wave.
//
// Run as separate kernels on separate streams, these steps do not overlap well: two attention
// CTAs fill an SM's shared memory and most of its registers, so a scoring or update CTA is placed
// only when the attention chain pauses, and the next layer's attention (launched early) takes the
// SMs first.  Here the CTAs take roles by index: the first n_attn CTAs are the attention split of
// the TMA kernel (its code, kvs_attn_tma.cuh); the next U * S CTAs score S tiles ranges of each
// unit (kvs_score.cuh); the last scoring CTA of a unit to finish (a per-unit counter, reset by
// it) selects the unit's top-K blocks and runs its cache update (kvs_select.cuh,
// kvs_update.cuh), which stages the new pending selection for the fetch that follows.  All roles
// use the same block size (the attention kernel's) and at most 160 registers per thread, so that a
// fetch CTA fits beside two of them.
#include "kvs_attn_tma.cuh"
#include "kvs_score.cuh"
#include "kvs_select.cuh"
#include "kvs_update.cuh"

#include <algorithm>

namespace kvs {

namespace {

constexpr int kLayerThreads = tma::kThreads;

struct LayerPlan {
  tma::Plan ap;          // the attention split over the first ap.n_cta CTAs
  int score_ctas;        // scoring CTAs per unit (S)
  int tiles_per_cta;     // 16-block tiles per scoring CTA
};

template <int NT, bool FP8, int DK, int NP>
__global__ void __maxnreg__(160)
    layer_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, Dims d, Layer L,
                 const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ index,
                 const __nv_bfloat16* __restrict__ sq, int nq, const int* __restrict__ ctx_len,
                 float* __restrict__ out, int* sel, int* nsel, kvs_stats* stats, LayerPlan lp) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ TopkShared tsh;
  __shared__ UpdateShared ush;
  __shared__ int s_last;
  if ((int)blockIdx.x < lp.ap.n_cta) {
    tma::attn_tma_cta<NT, FP8>(tmK, tmV, d, L, q, L.pend_sel, L.pend_slot, L.pend_n, ctx_len, out, lp.ap, blockIdx.x,
                               smem_raw);
    return;
  }
  const int j = blockIdx.x - lp.ap.n_cta;
  const int u = j / lp.score_ctas, bx = j % lp.score_ctas;
  kvs_pdl_entry();
  score_cta<DK, NP>(d, index, sq, nq, ctx_len, L.scores, lp.tiles_per_cta, L.err, bx, u, smem_raw);
  // the scores of this CTA are visible before it is counted; the last scoring CTA of the unit
  // selects and updates
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    s_last = atomicAdd(&L.score_done[u], 1u) == (unsigned)(lp.score_ctas - 1);
    if (s_last) L.score_done[u] = 0u;   // every scoring CTA of the unit has counted
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // one round of reads: the score row and every update input that does not depend on the selection
  UpdateIn in = update_stage(d, L, u, ctx_len, smem_raw, ush);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + select_keys_offset(d));
  topk_stage(d, L.scores, in.len, u, keys);
  cp_async_wait_all();
  __syncthreads();
  in.n = topk_staged(d, in.len, u, sel, nsel, L.err, keys, update_sel_buffer(d, smem_raw), tsh,
                     reinterpret_cast<uint32_t*>(smem_raw + select_scratch_offset(d)));
  __syncthreads();
  update_run(d, L, u, in, L.slot_of_sel, d.evict_importance ? L.scores : nullptr, stats, smem_raw, ush);
}

// Scoring CTAs per unit: the scoring share of one wave (2 CTAs per SM) in proportion to the bytes
// each role reads (index rows vs. K/V tiles), at least 1; the attention keeps at least half of
// the wave.
LayerPlan layer_plan(const Dims& d) {
  const int wave = 2 * device_sm_count();
  const double score_bytes = (double)d.U * d.nb_max * d.didx * 2.0;
  const double attn_bytes = (double)d.U * d.Kb * d.bs * (d.dk + d.dv) * d.ebytes;
  const int max_tiles = (d.nb_max + 15) / 16;
  int S = (int)(wave * score_bytes / (score_bytes + attn_bytes) / d.U + 0.5);
  S = std::max(1, std::min(S, max_tiles));
  while (S > 1 && d.U * S > wave / 2) --S;
  LayerPlan lp;
  lp.score_ctas = S;
  lp.tiles_per_cta = (max_tiles + S - 1) / S;
  lp.ap = tma::make_plan_ctas(d, wave - d.U * S);
  return lp;
}

template <int DK, int NP>
size_t layer_score_smem() {
  ScoreSmem sm{NP * 8, DK * 2 + 16, kLayerThreads / 32, score_stages<DK>()};
  return sm.bytes();
}

}  // namespace

int layer_kernel_supported(const Dims& d, int nq, bool have_tmaps) {
  if (!d.lookahead || !have_tmaps || !attention_tma_supported(d) || d.G > 8) return 0;
  if (!select_update_fusable(d) || score_tc_supported(d, nq)) return 0;
  if (d.didx != 128 && d.didx != 256) return 0;
  if (nq < 1 || nq * d.G > 32) return 0;
  return d.U <= device_sm_count();   // the attention keeps at least half of the wave
}

cudaError_t launch_layer(const Dims& d, const Layer& L, const __nv_bfloat16* q, const __nv_bfloat16* index,
                         const __nv_bfloat16* sq, int nq, const int* ctx_len, float* out, int* sel, int* nsel,
                         kvs_stats* stats, cudaStream_t s) {
  if (!layer_kernel_supported(d, nq, L.tmK && L.tmV)) return cudaErrorInvalidValue;
  const LayerPlan lp = layer_plan(d);
  const int grid = lp.ap.n_cta + d.U * lp.score_ctas;
  const size_t sel_smem = select_update_smem_bytes(d);
  auto go = [&](auto kern, size_t attn_smem, size_t score_smem) {
    const size_t smem = std::max(attn_smem, std::max(score_smem, sel_smem));
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kLayerThreads), smem, s, *L.tmK, *L.tmV, d, L, q, index, sq, nq, ctx_len,
                      out, sel, nsel, stats, lp);
  };
  const int np = nq * d.G <= 16 ? 2 : 4;
  cudaError_t e;
  if (d.fp8) {
    const size_t as = tma::Smem<1, true>::bytes(d.G, lp.ap.per_cta);
    if (d.didx == 128)
      e = np == 2 ? go(layer_kernel<1, true, 128, 2>, as, layer_score_smem<128, 2>())
                  : go(layer_kernel<1, true, 128, 4>, as, layer_score_smem<128, 4>());
    else
      e = np == 2 ? go(layer_kernel<1, true, 256, 2>, as, layer_score_smem<256, 2>())
                  : go(layer_kernel<1, true, 256, 4>, as, layer_score_smem<256, 4>());
  } else {
    const size_t as = tma::Smem<1, false>::bytes(d.G, lp.ap.per_cta);
    if (d.didx == 128)
      e = np == 2 ? go(layer_kernel<1, false, 128, 2>, as, layer_score_smem<128, 2>())
                  : go(layer_kernel<1, false, 128, 4>, as, layer_score_smem<128, 4>());
    else
      e = np == 2 ? go(layer_kernel<1, false, 256, 2>, as, layer_score_smem<256, 2>())
                  : go(layer_kernel<1, false, 256, 4>, as, layer_score_smem<256, 4>());
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvs
