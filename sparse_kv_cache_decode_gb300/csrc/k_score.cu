// Block scoring: s[b] = scale * max over the unit's scoring rows r of (q_r . ik[b]).
//
// Tensor-core tile (m16n8k16, bf16 in, fp32 accumulate): A = 16 index keys (blocks) x 16 dims,
// B = 16 dims x 8 scoring rows.  The scoring rows of unit (request, kv-head h) are the q heads
// of group h for every scoring query j (row = j * G + g).  Rows are kept in shared memory for the
// whole CTA; index tiles stream through a per-warp ring of cp.async stages (4 for rows of up to
// 256 bytes, 2 for wider rows).  The max over rows is taken in registers and across the 4 lanes
// of a quad.  The grid is one wave: the CTAs per unit are chosen from the resident CTAs per SM.
#include <float.h>

#include "kvs_common.cuh"
#include "kvs_ptx.cuh"

namespace kvs {

namespace {

constexpr int kScoreMaxRows = 128;

template <int DK>
constexpr int score_stages() { return DK <= 128 ? 4 : 2; }

struct ScoreSmem {
  int rows_pad;     // scoring rows rounded up to 16
  int row_stride;   // bytes per smem row (dk * 2 + 16 pad: conflict-free ldmatrix)
  int nwarps;
  int stages;
  size_t bytes() const { return (size_t)rows_pad * row_stride + (size_t)nwarps * stages * 16 * row_stride; }
};

template <int DK, int NP>  // DK = index row width d_idx; NP = number of n8 tiles of scoring rows (rows_pad / 8)
__global__ void __launch_bounds__(128) score_kernel(Dims d, const __nv_bfloat16* __restrict__ index,
                                                    const __nv_bfloat16* __restrict__ q, int nq,
                                                    const int* __restrict__ ctx_len, float* __restrict__ scores,
                                                    int tiles_per_cta, unsigned* err) {
  kvs_pdl_entry();
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int RS = DK * 2 + 16;  // row stride in bytes
  constexpr int KSTEPS = DK / 16;
  constexpr int CH = DK * 2 / 16;  // 16-byte chunks per row
  const int u = blockIdx.y;
  const int r = u / d.Hkv, h = u % d.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int len = ctx_len[r];
  if (len < 0 || len > d.max_ctx) {
    if (threadIdx.x == 0) set_error(err, KVS_ERR_BAD_INDEX);
    return;
  }
  const int nb = n_blocks_of(len, d.bs);
  const int n_tiles = (nb + 15) / 16;
  const int tile0 = blockIdx.x * tiles_per_cta;
  const int tile1 = min(n_tiles, tile0 + tiles_per_cta);
  if (tile0 >= tile1) return;
  const int R = nq * d.G;

  // scoring rows -> smem (zero rows beyond R)
  unsigned char* qs = smem;
  for (int i = threadIdx.x; i < NP * 8 * CH; i += blockDim.x) {
    int row = i / CH, ch = i % CH;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < R) {
      int j = row / d.G, g = row % d.G;
      v = score_row_chunk(q + (((size_t)r * nq + j) * d.Hq + h * d.G + g) * d.dk, ch, d);
    }
    *reinterpret_cast<uint4*>(qs + row * RS + ch * 16) = v;
  }
  __syncthreads();

  constexpr int ST = score_stages<DK>();
  unsigned char* buf = smem + NP * 8 * RS + (size_t)warp * ST * 16 * RS;
  const __nv_bfloat16* ik = index + (size_t)u * d.nb_max * DK;

  auto load_tile = [&](int tile, int stage) {
    unsigned char* dst = buf + stage * 16 * RS;
    for (int i = lane; i < 16 * CH; i += 32) {
      int row = i / CH, ch = i % CH;
      int b = tile * 16 + row;
      const __nv_bfloat16* src = ik + (size_t)min(b, nb - 1) * DK + ch * 8;
      cp_async16(dst + row * RS + ch * 16, src, b < nb ? 16 : 0);
    }
    cp_async_commit();
  };

  // ring of ST stages: tiles my, my + nwarps, ... ; ST - 1 loads stay in flight ahead of the one
  // being computed (an empty group is committed past the end so the wait count stays fixed)
  const int first = tile0 + warp;
#pragma unroll
  for (int i = 0; i < ST - 1; ++i) {
    const int t = first + i * nwarps;
    if (t < tile1) load_tile(t, i);
    else cp_async_commit();
  }
  int stage = 0;
  for (int my = first; my < tile1; my += nwarps, stage = (stage + 1) % ST) {
    const int ahead = my + (ST - 1) * nwarps;
    if (ahead < tile1) load_tile(ahead, (stage + ST - 1) % ST);
    else cp_async_commit();
    cp_async_wait<ST - 1>();
    __syncwarp();
    const unsigned char* a_tile = buf + stage * 16 * RS;
    float acc[NP][4];
#pragma unroll
    for (int n = 0; n < NP; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      uint32_t a0, a1, a2, a3;
      // matrices: (rows 0-7, k 0-7), (rows 8-15, k 0-7), (rows 0-7, k 8-15), (rows 8-15, k 8-15)
      {
        int mrow = (lane & 7) + ((lane >> 3) & 1) * 8;
        int kcol = ks * 16 + (lane >> 4) * 8;
        ldmatrix_x4(a0, a1, a2, a3, a_tile + mrow * RS + kcol * 2);
      }
#pragma unroll
      for (int n = 0; n < NP; n += 2) {
        if (n + 1 < NP) {
          uint32_t b0, b1, b2, b3;
          // matrices: (rows n0..+7, k 0-7), (rows n0..+7, k 8-15), (rows n0+8.., k 0-7), (rows n0+8.., k 8-15)
          int qrow = n * 8 + (lane & 7) + (lane >> 4) * 8;
          int kcol = ks * 16 + ((lane >> 3) & 1) * 8;
          ldmatrix_x4(b0, b1, b2, b3, qs + qrow * RS + kcol * 2);
          mma_bf16_16816(acc[n], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(acc[n + 1], a0, a1, a2, a3, b2, b3);
        } else {
          uint32_t b0, b1;
          int qrow = n * 8 + (lane & 7);
          int kcol = ks * 16 + ((lane >> 3) & 1) * 8;
          ldmatrix_x2(b0, b1, qs + qrow * RS + kcol * 2);
          mma_bf16_16816(acc[n], a0, a1, a2, a3, b0, b1);
        }
      }
    }
    __syncwarp();   // the stage is refilled only after every lane has read it
    // max over valid scoring rows (columns)
    float m_lo = -FLT_MAX, m_hi = -FLT_MAX;
#pragma unroll
    for (int n = 0; n < NP; ++n) {
      int c0 = n * 8 + (lane & 3) * 2;
      if (c0 < R) { m_lo = fmaxf(m_lo, acc[n][0]); m_hi = fmaxf(m_hi, acc[n][2]); }
      if (c0 + 1 < R) { m_lo = fmaxf(m_lo, acc[n][1]); m_hi = fmaxf(m_hi, acc[n][3]); }
    }
    m_lo = fmaxf(m_lo, __shfl_xor_sync(0xffffffffu, m_lo, 1));
    m_lo = fmaxf(m_lo, __shfl_xor_sync(0xffffffffu, m_lo, 2));
    m_hi = fmaxf(m_hi, __shfl_xor_sync(0xffffffffu, m_hi, 1));
    m_hi = fmaxf(m_hi, __shfl_xor_sync(0xffffffffu, m_hi, 2));
    if ((lane & 3) == 0) {
      int b_lo = my * 16 + (lane >> 2), b_hi = b_lo + 8;
      float* out = scores + (size_t)u * d.nb_max;
      if (b_lo < nb) out[b_lo] = __fmul_rn(d.scale, m_lo);
      if (b_hi < nb) out[b_hi] = __fmul_rn(d.scale, m_hi);
    }
  }
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
