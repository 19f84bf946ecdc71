// Block scoring by one CTA: s[b] = scale * max over the unit's scoring rows r of (q_r . ik[b]).
//
// Tensor-core tile (m16n8k16, bf16 in, fp32 accumulate): A = 16 index keys (blocks) x 16 dims,
// B = 16 dims x 8 scoring rows.  The scoring rows of unit (request, kv-head h) are the q heads
// of group h for every scoring query j (row = j * G + g).  Rows are kept in shared memory for the
// whole CTA; index tiles stream through a per-warp ring of cp.async stages (4 for rows of up to
// 256 bytes, 2 for wider rows).  The max over rows is taken in registers and across the 4 lanes
// of a quad.  Shared by the scoring kernel and the fused layer kernel.
#pragma once
#include <float.h>

#include "kvs_common.cuh"
#include "kvs_ptx.cuh"

namespace kvs {

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

// Scores of tiles [bx * tiles_per_cta, (bx + 1) * tiles_per_cta) of unit u by one CTA (every thread
// of the CTA calls it; the warps share the work).  smem: ScoreSmem bytes, 16-byte aligned.
template <int DK, int NP>  // DK = index row width d_idx; NP = number of n8 tiles of scoring rows (rows_pad / 8)
__device__ inline void score_cta(const Dims& d, const __nv_bfloat16* __restrict__ index,
                                 const __nv_bfloat16* __restrict__ q, int nq, const int* __restrict__ ctx_len,
                                 float* __restrict__ scores, int tiles_per_cta, unsigned* err, int bx, int u,
                                 unsigned char* smem) {
  constexpr int RS = DK * 2 + 16;  // row stride in bytes
  constexpr int KSTEPS = DK / 16;
  constexpr int CH = DK * 2 / 16;  // 16-byte chunks per row
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
  const int tile0 = bx * tiles_per_cta;
  const int tile1 = min(n_tiles, tile0 + tiles_per_cta);
  if (tile0 >= tile1) return;
  const int R = nq * d.G;

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
  // being computed (an empty group is committed past the end so the wait count stays fixed).  The
  // first loads are issued before the scoring rows are staged, so that their latency overlaps it.
  const int first = tile0 + warp;
#pragma unroll
  for (int i = 0; i < ST - 1; ++i) {
    const int t = first + i * nwarps;
    if (t < tile1) load_tile(t, i);
    else cp_async_commit();
  }
  // scoring rows -> smem (zero rows beyond R); the ring buffers lie after them
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

}  // namespace kvs
