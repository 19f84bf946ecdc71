// Block scoring: s[b] = scale * max over the unit's scoring rows r of (q_r . ik[b]).
//
// Tensor-core tile (m16n8k16, bf16 in, fp32 accumulate): A = 16 index keys (blocks) x 16 dims,
// B = 16 dims x 8 scoring rows.  The scoring rows of unit (request, kv-head h) are the q heads
// of group h for every scoring query j (row = j * G + g).  Rows are kept in shared memory for the
// whole CTA; index tiles stream through a per-warp ring of cp.async stages (4 for rows of up to
// 256 bytes, 2 for wider rows).  The max over rows is taken in registers and across the 4 lanes
// of a quad.  The grid is one wave: the CTAs per unit are chosen from the resident CTAs per SM.
#include "kvs_common.cuh"
#include "kvs_ptx.cuh"
#include "kvs_score.cuh"

namespace kvs {

namespace {

template <int DK, int NP>
__global__ void __launch_bounds__(128) score_kernel(Dims d, const __nv_bfloat16* __restrict__ index,
                                                    const __nv_bfloat16* __restrict__ q, int nq,
                                                    const int* __restrict__ ctx_len, float* __restrict__ scores,
                                                    int tiles_per_cta, unsigned* err) {
  kvs_pdl_entry();
  extern __shared__ __align__(16) unsigned char smem[];
  score_cta<DK, NP>(d, index, q, nq, ctx_len, scores, tiles_per_cta, err, blockIdx.x, blockIdx.y, smem);
}

template <int DK, int NP>
cudaError_t launch_score_t(const Dims& d, const __nv_bfloat16* index, const __nv_bfloat16* q, int nq,
                           const int* ctx_len, float* scores, unsigned* err, cudaStream_t s) {
  constexpr int ST = score_stages<DK>();
  int nwarps = (DK * 2 + 16) * (NP * 8 + 4 * ST * 16) <= 200 * 1024 ? 4 : 2;
  ScoreSmem sm{NP * 8, DK * 2 + 16, nwarps, ST};
  size_t bytes = sm.bytes();
  auto kern = score_kernel<DK, NP>;
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), (int)bytes);
    if (e != cudaSuccess) return e;
  }
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * nwarps, bytes) != cudaSuccess || per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  int max_tiles = (d.nb_max + 15) / 16;
  // one wave of CTAs over the SMs, at least 4 tiles per warp
  int ctas_per_unit = max(1, min((max_tiles + 4 * nwarps - 1) / (4 * nwarps), per_sm * device_sm_count() / d.U));
  int tiles_per_cta = (max_tiles + ctas_per_unit - 1) / ctas_per_unit;
  dim3 grid(ctas_per_unit, d.U);
  launch_pdl(kern, dim3(grid), dim3(32 * nwarps), bytes, s, d, index, q, nq, ctx_len, scores, tiles_per_cta, err);
  return cudaGetLastError();
}

}  // namespace

int score_supported(const Dims& d) {
  // every call width 1..max_nq must have a kernel: tcgen05 for wide rows, mma.sync otherwise
  for (int nq = 1; nq <= d.max_nq; ++nq) {
    const bool mma = (d.didx == 128 || d.didx == 256 || d.didx == 576) && nq * d.G <= kScoreMaxRows;
    if (!mma && !score_tc_supported(d, nq)) return 0;
  }
  return 1;
}

cudaError_t launch_score(const Dims& d, const __nv_bfloat16* index, const __nv_bfloat16* q, int nq,
                             const int* ctx_len, float* scores, unsigned* err, cudaStream_t s) {
  if (score_tc_supported(d, nq)) return launch_score_tc(d, index, q, nq, ctx_len, scores, err, s);
  int R = nq * d.G;
  int np = (R + 7) / 8;
  if (np > 16 || nq < 1) return cudaErrorInvalidValue;
  np = np <= 2 ? 2 : np <= 4 ? 4 : np <= 8 ? 8 : 16;  // padded rows are zero and masked out
  if (d.didx == 128) {
    switch (np) {
      case 2: return launch_score_t<128, 2>(d, index, q, nq, ctx_len, scores, err, s);
      case 4: return launch_score_t<128, 4>(d, index, q, nq, ctx_len, scores, err, s);
      case 8: return launch_score_t<128, 8>(d, index, q, nq, ctx_len, scores, err, s);
      case 16: return launch_score_t<128, 16>(d, index, q, nq, ctx_len, scores, err, s);
      default: break;
    }
  } else if (d.didx == 256) {
    switch (np) {
      case 2: return launch_score_t<256, 2>(d, index, q, nq, ctx_len, scores, err, s);
      case 4: return launch_score_t<256, 4>(d, index, q, nq, ctx_len, scores, err, s);
      case 8: return launch_score_t<256, 8>(d, index, q, nq, ctx_len, scores, err, s);
      case 16: return launch_score_t<256, 16>(d, index, q, nq, ctx_len, scores, err, s);
      default: break;
    }
  } else if (d.didx == 576) {
    switch (np) {
      case 2: return launch_score_t<576, 2>(d, index, q, nq, ctx_len, scores, err, s);
      case 4: return launch_score_t<576, 4>(d, index, q, nq, ctx_len, scores, err, s);
      case 8: return launch_score_t<576, 8>(d, index, q, nq, ctx_len, scores, err, s);
      case 16: return launch_score_t<576, 16>(d, index, q, nq, ctx_len, scores, err, s);
      default: break;
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvs
