// Exact decode attention over the selected cache slots of each unit.
//
// Grid (split, unit, dv-chunk).  A CTA takes a contiguous range of the unit's selected blocks,
// walks their present tokens in 16-token tiles staged in shared memory by cp.async, and keeps
// an online softmax per q head.  Tensor-core tiles (m16n8k16, bf16 in, fp32 accumulate):
//   S  = Q (16 heads x d_k) . K^T (d_k x 16 tokens)
//   O += P (16 heads x 16 tokens) . V (16 tokens x 8-dim tiles); V fragments via ldmatrix.trans;
//   P is split into bf16 high and low parts (two products) so it keeps ~16 bits.
// With G <= 16 one 16-row head tile covers the group and the CTA's warps split the tiles
// (their partial softmax states are merged in shared memory); with larger G each warp owns a
// 16-head tile and all warps read every token tile.  V is split into 128-wide chunks across
// the grid's z dimension so the accumulators stay in registers.  Partial results of the
// splits are merged by a second kernel: o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
#include <float.h>

#include "kvs_common.cuh"
#include "kvs_ptx.cuh"

namespace kvs {

namespace {

constexpr int kDVC = 128;              // V columns per CTA
constexpr float kLog2e = 1.4426950408889634f;

template <int DK, int MT, bool VSHARE>
struct AttnCfg {
  static constexpr int NW = MT == 1 ? 4 : MT;           // warps
  static constexpr int KRS = DK * 2 + 16;               // K tile row stride (bytes)
  static constexpr int VRS = kDVC * 2 + 16;             // V tile row stride (bytes)
  static constexpr int TILE_BYTES = 16 * KRS + (VSHARE ? 0 : 16 * VRS);
  static constexpr int NBUF = MT == 1 ? NW * 2 : 2;     // per-warp double buffers, or shared
  static constexpr int Q_BYTES = MT * 16 * KRS;
  static constexpr int BUF_BYTES = NBUF * TILE_BYTES;
  static constexpr int COMB_BYTES = MT == 1 ? NW * 16 * (kDVC + 2) * 4 : 0;
  static constexpr int SMEM = Q_BYTES + (BUF_BYTES > COMB_BYTES ? BUF_BYTES : COMB_BYTES) + 4 * 1024;
};

template <int DK, int MT, bool VSHARE>
__global__ void __launch_bounds__(AttnCfg<DK, MT, VSHARE>::NW * 32)
    attn_kernel(Dims d, Layer L, const __nv_bfloat16* __restrict__ q, const int* __restrict__ sel,
                const int* __restrict__ slot_of_sel, const int* __restrict__ nsel, const int* __restrict__ ctx_len,
                float* __restrict__ out, int n_split, int blocks_per_split) {
  kvs_pdl_entry();
  using Cfg = AttnCfg<DK, MT, VSHARE>;
  constexpr int NW = Cfg::NW, KRS = Cfg::KRS, VRS = Cfg::VRS;
  constexpr int KSTEPS = DK / 16;
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* qs = smem;
  unsigned char* bufs = smem + Cfg::Q_BYTES;
  const int max_blocks_cta = (Cfg::SMEM - Cfg::Q_BYTES - (Cfg::BUF_BYTES > Cfg::COMB_BYTES ? Cfg::BUF_BYTES : Cfg::COMB_BYTES)) / 8;
  int* s_slot = reinterpret_cast<int*>(bufs + (Cfg::BUF_BYTES > Cfg::COMB_BYTES ? Cfg::BUF_BYTES : Cfg::COMB_BYTES));
  int* s_blk = s_slot + max_blocks_cta;

  const int split = blockIdx.x, u = blockIdx.y, z = blockIdx.z;
  const int r = u / d.Hkv, h = u % d.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int len = ctx_len[r];
  int n = nsel[u];
  if (len < 0 || len > d.max_ctx || n < 0 || n > d.Kb) {   // reported; the unit attends to nothing
    if (tid == 0) set_error(L.err, KVS_ERR_BAD_INDEX);
    len = 0;
    n = 0;
  }
  const int i0 = min(n, split * blocks_per_split), i1 = min(n, i0 + blocks_per_split);
  const int nblk = i1 - i0;
  const int n_tok = nblk * d.bs;
  const int n_tiles = (n_tok + 15) / 16;
  const int G = d.G;
  const int dv0 = z * kDVC;

  // queries of the group -> smem (rows >= G zero)
  for (int i = tid; i < MT * 16 * (DK / 8); i += NW * 32) {
    int row = i / (DK / 8), ch = i % (DK / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < G) v = reinterpret_cast<const uint4*>(q + ((size_t)r * d.Hq + h * G + row) * DK)[ch];
    *reinterpret_cast<uint4*>(qs + row * KRS + ch * 16) = v;
  }
  for (int i = tid; i < nblk; i += NW * 32) {
    int slot = slot_of_sel[(size_t)u * d.Kb + i0 + i];
    int blk = sel[(size_t)u * d.Kb + i0 + i];
    if (blk < 0 || blk >= n_blocks_of(len, d.bs) || slot < 0 || slot >= d.C) {   // reported, then masked
      set_error(L.err, KVS_ERR_BAD_INDEX);
      slot = -1;
      blk = 0;
    }
    s_slot[i] = slot;
    s_blk[i] = blk;
  }
  __syncthreads();

  const __nv_bfloat16* kbase = L.kpool + (size_t)u * d.C * d.bs * DK;
  const __nv_bfloat16* vbase = VSHARE ? kbase : L.vpool + (size_t)u * d.C * d.bs * d.dv;

  // token k of this CTA -> (block, row); valid when inside the range and before len
  auto tok_ptr = [&](int k, bool& valid, size_t& row_index) {
    int bi = k / d.bs, rr = k - bi * d.bs;
    valid = false;
    row_index = 0;
    if (bi < nblk) {
      int pos = s_blk[bi] * d.bs + rr;
      int slot = s_slot[bi];
      valid = pos < len && slot >= 0 && slot < d.C;
      row_index = valid ? (size_t)slot * d.bs + rr : 0;
    }
  };

  // stage tile t (16 tokens) into buffer `dst` using `nthreads` threads starting at `t0`
  auto load_tile = [&](int t, unsigned char* dst, int t_first, int nthreads) {
    constexpr int KCH = DK * 2 / 16;
    constexpr int VCH = kDVC * 2 / 16;
    for (int i = t_first; i < 16 * KCH; i += nthreads) {
      int row = i / KCH, ch = i % KCH;
      bool valid;
      size_t ri;
      tok_ptr(t * 16 + row, valid, ri);
      const __nv_bfloat16* src = kbase + ri * DK + ch * 8;
      cp_async16(dst + row * KRS + ch * 16, valid ? (const void*)src : (const void*)kbase, valid ? 16 : 0);
    }
    if (!VSHARE) {
      unsigned char* vdst = dst + 16 * KRS;
      for (int i = t_first; i < 16 * VCH; i += nthreads) {
        int row = i / VCH, ch = i % VCH;
        bool valid;
        size_t ri;
        tok_ptr(t * 16 + row, valid, ri);
        const __nv_bfloat16* src = vbase + ri * d.dv + dv0 + ch * 8;
        cp_async16(vdst + row * VRS + ch * 16, valid ? (const void*)src : (const void*)vbase, valid ? 16 : 0);
      }
    }
    cp_async_commit();
  };

  const int ht = MT == 1 ? 0 : warp;  // head tile of this warp
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  float oacc[kDVC / 8][4];
#pragma unroll
  for (int i = 0; i < kDVC / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  const float sl2 = d.scale * kLog2e;

  auto process_tile = [&](int t, const unsigned char* tile) {
    const unsigned char* kt = tile;
    const unsigned char* vt = VSHARE ? tile : tile + 16 * KRS;
    const int vrs = VSHARE ? KRS : VRS;
    const int vcol0 = VSHARE ? dv0 : 0;
    float sacc[2][4];
#pragma unroll
    for (int nn = 0; nn < 2; ++nn) sacc[nn][0] = sacc[nn][1] = sacc[nn][2] = sacc[nn][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
      {
        int mrow = ht * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        int kcol = ks * 16 + (lane >> 4) * 8;
        ldmatrix_x4(a0, a1, a2, a3, qs + mrow * KRS + kcol * 2);
      }
      {
        int trow = (lane & 7) + (lane >> 4) * 8;
        int kcol = ks * 16 + ((lane >> 3) & 1) * 8;
        ldmatrix_x4(b0, b1, b2, b3, kt + trow * KRS + kcol * 2);
      }
      mma_bf16_16816(sacc[0], a0, a1, a2, a3, b0, b1);
      mma_bf16_16816(sacc[1], a0, a1, a2, a3, b2, b3);
    }
    // scale (log2 domain) and mask
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int nn = 0; nn < 2; ++nn) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        int k = t * 16 + nn * 8 + (lane & 3) * 2 + e;
        bool valid;
        size_t ri;
        tok_ptr(k, valid, ri);
        float s_lo = valid ? sacc[nn][e] * sl2 : -INFINITY;
        float s_hi = valid ? sacc[nn][2 + e] * sl2 : -INFINITY;
        sacc[nn][e] = s_lo;
        sacc[nn][2 + e] = s_hi;
        mx_lo = fmaxf(mx_lo, s_lo);
        mx_hi = fmaxf(mx_hi, s_hi);
      }
    }
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float al_lo = mn_lo == -INFINITY ? 1.f : exp2f(m_lo - mn_lo);
    const float al_hi = mn_hi == -INFINITY ? 1.f : exp2f(m_hi - mn_hi);
    float ps_lo = 0.f, ps_hi = 0.f;
#pragma unroll
    for (int nn = 0; nn < 2; ++nn) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float p_lo = mn_lo == -INFINITY ? 0.f : exp2f(sacc[nn][e] - mn_lo);
        float p_hi = mn_hi == -INFINITY ? 0.f : exp2f(sacc[nn][2 + e] - mn_hi);
        sacc[nn][e] = p_lo;
        sacc[nn][2 + e] = p_hi;
        ps_lo += p_lo;
        ps_hi += p_hi;
      }
    }
    ps_lo += __shfl_xor_sync(0xffffffffu, ps_lo, 1);
    ps_lo += __shfl_xor_sync(0xffffffffu, ps_lo, 2);
    ps_hi += __shfl_xor_sync(0xffffffffu, ps_hi, 1);
    ps_hi += __shfl_xor_sync(0xffffffffu, ps_hi, 2);
    l_lo = l_lo * al_lo + ps_lo;
    l_hi = l_hi * al_hi + ps_hi;
    m_lo = mn_lo;
    m_hi = mn_hi;
    // P = P_hi + P_lo with both parts bf16: two products keep P to ~2^-16 relative
    uint32_t ph[4], pl[4];
    auto split2 = [](float a, float b, uint32_t& hi, uint32_t& lo) {
      hi = pack_bf16x2(a, b);
      lo = pack_bf16x2(a - bf16_lo(hi), b - bf16_hi(hi));
    };
    split2(sacc[0][0], sacc[0][1], ph[0], pl[0]);
    split2(sacc[0][2], sacc[0][3], ph[1], pl[1]);
    split2(sacc[1][0], sacc[1][1], ph[2], pl[2]);
    split2(sacc[1][2], sacc[1][3], ph[3], pl[3]);
#pragma unroll
    for (int nd = 0; nd < kDVC / 8; nd += 2) {
      oacc[nd][0] *= al_lo; oacc[nd][1] *= al_lo; oacc[nd][2] *= al_hi; oacc[nd][3] *= al_hi;
      oacc[nd + 1][0] *= al_lo; oacc[nd + 1][1] *= al_lo; oacc[nd + 1][2] *= al_hi; oacc[nd + 1][3] *= al_hi;
      uint32_t b0, b1, b2, b3;
      int trow = (lane & 7) + ((lane >> 3) & 1) * 8;
      int col = vcol0 + nd * 8 + (lane >> 4) * 8;
      ldmatrix_x4_trans(b0, b1, b2, b3, vt + trow * vrs + col * 2);
      mma_bf16_16816(oacc[nd], ph[0], ph[1], ph[2], ph[3], b0, b1);
      mma_bf16_16816(oacc[nd], pl[0], pl[1], pl[2], pl[3], b0, b1);
      mma_bf16_16816(oacc[nd + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
      mma_bf16_16816(oacc[nd + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
    }
  };

  if (MT == 1) {
    // warps split the tiles; each warp double-buffers its own tiles
    unsigned char* mybuf = bufs + (size_t)warp * 2 * Cfg::TILE_BYTES;
    int t = warp, stage = 0;
    if (t < n_tiles) load_tile(t, mybuf, lane, 32);
    for (; t < n_tiles; t += NW, stage ^= 1) {
      int nt = t + NW;
      if (nt < n_tiles) { load_tile(nt, mybuf + (stage ^ 1) * Cfg::TILE_BYTES, lane, 32); cp_async_wait<1>(); }
      else cp_async_wait<0>();
      __syncwarp();
      process_tile(t, mybuf + stage * Cfg::TILE_BYTES);
      __syncwarp();
    }
  } else {
    int stage = 0;
    if (n_tiles > 0) load_tile(0, bufs, tid, NW * 32);
    for (int t = 0; t < n_tiles; ++t, stage ^= 1) {
      if (t + 1 < n_tiles) { load_tile(t + 1, bufs + (stage ^ 1) * Cfg::TILE_BYTES, tid, NW * 32); cp_async_wait<1>(); }
      else cp_async_wait<0>();
      __syncthreads();
      process_tile(t, bufs + stage * Cfg::TILE_BYTES);
      __syncthreads();
    }
  }

  // rows of this thread: head ht*16 + lane/4 (lo) and +8 (hi); columns nd*8 + 2*(lane%4) + {0,1}
  const int row_lo = ht * 16 + (lane >> 2), row_hi = row_lo + 8;
  float* part = L.attn_part;
  float* pml = L.attn_ml;

  if (MT == 1) {
    // merge the warps' states in shared memory
    __syncthreads();
    float* cb = reinterpret_cast<float*>(bufs);                 // [NW][16][kDVC]
    float* cm = cb + NW * 16 * kDVC;                            // [NW][16][2]
#pragma unroll
    for (int nd = 0; nd < kDVC / 8; ++nd) {
      int c = nd * 8 + (lane & 3) * 2;
      cb[(warp * 16 + (lane >> 2)) * kDVC + c] = oacc[nd][0];
      cb[(warp * 16 + (lane >> 2)) * kDVC + c + 1] = oacc[nd][1];
      cb[(warp * 16 + (lane >> 2) + 8) * kDVC + c] = oacc[nd][2];
      cb[(warp * 16 + (lane >> 2) + 8) * kDVC + c + 1] = oacc[nd][3];
    }
    if ((lane & 3) == 0) {
      cm[(warp * 16 + (lane >> 2)) * 2 + 0] = m_lo;
      cm[(warp * 16 + (lane >> 2)) * 2 + 1] = l_lo;
      cm[(warp * 16 + (lane >> 2) + 8) * 2 + 0] = m_hi;
      cm[(warp * 16 + (lane >> 2) + 8) * 2 + 1] = l_hi;
    }
    __syncthreads();
    for (int i = tid; i < G * kDVC; i += NW * 32) {
      int row = i / kDVC, c = i % kDVC;
      float M = -INFINITY;
      for (int w = 0; w < NW; ++w) M = fmaxf(M, cm[(w * 16 + row) * 2]);
      float o = 0.f, lsum = 0.f;
      if (M != -INFINITY) {
        for (int w = 0; w < NW; ++w) {
          float mw = cm[(w * 16 + row) * 2];
          float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
          o += f * cb[(w * 16 + row) * kDVC + c];
          lsum += f * cm[(w * 16 + row) * 2 + 1];
        }
      }
      if (n_split == 1) {
        out[((size_t)r * d.Hq + h * G + row) * d.dv + dv0 + c] = lsum > 0.f ? o / lsum : 0.f;
      } else {
        part[(((size_t)u * n_split + split) * G + row) * d.dv + dv0 + c] = o;
        if (c == 0 && z == 0) {
          pml[(((size_t)u * n_split + split) * G + row) * 2 + 0] = M;
          pml[(((size_t)u * n_split + split) * G + row) * 2 + 1] = lsum;
        }
      }
    }
  } else {
    // each warp owns its rows
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int row = hh ? row_hi : row_lo;
      const float m = hh ? m_hi : m_lo, l = hh ? l_hi : l_lo;
      if (row >= G) continue;
#pragma unroll
      for (int nd = 0; nd < kDVC / 8; ++nd) {
        int c = nd * 8 + (lane & 3) * 2;
        float o0 = oacc[nd][hh * 2], o1 = oacc[nd][hh * 2 + 1];
        if (n_split == 1) {
          float* dst = out + ((size_t)r * d.Hq + h * G + row) * d.dv + dv0 + c;
          dst[0] = l > 0.f ? o0 / l : 0.f;
          dst[1] = l > 0.f ? o1 / l : 0.f;
        } else {
          float* dst = part + (((size_t)u * n_split + split) * G + row) * d.dv + dv0 + c;
          dst[0] = o0;
          dst[1] = o1;
        }
      }
      if (n_split > 1 && z == 0 && (lane & 3) == 0) {
        pml[(((size_t)u * n_split + split) * G + row) * 2 + 0] = m;
        pml[(((size_t)u * n_split + split) * G + row) * 2 + 1] = l;
      }
    }
  }
}

// MLA decode attention (d_k = 576 latent + rope dims, V = the first 512 dims of each K row,
// heads in groups of 32).  Grid (split, unit, head group).  The 8 warps are 2 head tiles x 4
// quarters: warp (ht, qq) computes the q.k product over dims [144 qq, 144 qq + 144) for its 16
// heads, the four partial 16 x 16 score tiles of a head tile are summed through shared memory
// in a fixed order (named barrier of the tile's 4 warps), then every warp runs the online
// softmax of its head tile and accumulates P.V for value columns [128 qq, 128 qq + 128).  So
// the q.k product is computed once per (head, token), and 32 heads of queries (36 KiB) leave
// room for two CTAs per SM.
namespace mla {
constexpr int DK = 576, DV = 512, HEADS = 32, NW = 8, QDIMS = DK / 4;
constexpr int KRS = DK * 2 + 16;                 // row stride of query and token rows (bytes)
constexpr int TILE = 16 * KRS;                   // 16 token rows
constexpr int Q_BYTES = HEADS * KRS;
constexpr int RED_BYTES = 2 * 4 * 256 * 4;       // [head tile][quarter][256 fragment floats]
constexpr int LIST_ENTRIES = 512;                // staged (block, slot) pairs per CTA
constexpr int SMEM = Q_BYTES + 2 * TILE + RED_BYTES + LIST_ENTRIES * 8;
}  // namespace mla

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

__global__ void __launch_bounds__(mla::NW * 32, 2)
    attn_mla_kernel(Dims d, Layer L, const __nv_bfloat16* __restrict__ q, const int* __restrict__ sel,
                    const int* __restrict__ slot_of_sel, const int* __restrict__ nsel,
                    const int* __restrict__ ctx_len, float* __restrict__ out, int n_split, int blocks_per_split) {
  kvs_pdl_entry();
  using namespace mla;
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* qs = smem;
  unsigned char* bufs = smem + Q_BYTES;
  float* red = reinterpret_cast<float*>(bufs + 2 * TILE);
  int* s_slot = reinterpret_cast<int*>(bufs + 2 * TILE + RED_BYTES);
  int* s_blk = s_slot + LIST_ENTRIES;

  const int split = blockIdx.x, u = blockIdx.y, hg = blockIdx.z;
  const int r = u / d.Hkv, h = u % d.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ht = warp >> 2, qq = warp & 3;
  int len = ctx_len[r];
  int n = nsel[u];
  if (len < 0 || len > d.max_ctx || n < 0 || n > d.Kb) {   // reported; the unit attends to nothing
    if (tid == 0) set_error(L.err, KVS_ERR_BAD_INDEX);
    len = 0;
    n = 0;
  }
  const int i0 = min(n, split * blocks_per_split), i1 = min(n, i0 + blocks_per_split);
  const int nblk = i1 - i0;
  const int n_tiles = (nblk * d.bs + 15) / 16;
  const int head0 = h * d.G + hg * HEADS;          // first q head of the CTA

  for (int i = tid; i < HEADS * (DK / 8); i += NW * 32) {
    const int row = i / (DK / 8), ch = i % (DK / 8);
    *reinterpret_cast<uint4*>(qs + row * KRS + ch * 16) =
        reinterpret_cast<const uint4*>(q + ((size_t)r * d.Hq + head0 + row) * DK)[ch];
  }
  for (int i = tid; i < nblk; i += NW * 32) {
    int slot = slot_of_sel[(size_t)u * d.Kb + i0 + i];
    int blk = sel[(size_t)u * d.Kb + i0 + i];
    if (blk < 0 || blk >= n_blocks_of(len, d.bs) || slot < 0 || slot >= d.C) {   // reported, then masked
      set_error(L.err, KVS_ERR_BAD_INDEX);
      slot = -1;
      blk = 0;
    }
    s_slot[i] = slot;
    s_blk[i] = blk;
  }
  __syncthreads();

  const __nv_bfloat16* kbase = L.kpool + (size_t)u * d.C * d.bs * DK;
  auto tok_ptr = [&](int k, bool& valid, size_t& row_index) {
    const int bi = k / d.bs, rr = k - bi * d.bs;
    valid = false;
    row_index = 0;
    if (bi < nblk) {
      const int pos = s_blk[bi] * d.bs + rr;
      const int slot = s_slot[bi];
      valid = pos < len && slot >= 0 && slot < d.C;
      row_index = valid ? (size_t)slot * d.bs + rr : 0;
    }
  };
  auto load_tile = [&](int t, unsigned char* dst) {
    constexpr int KCH = DK * 2 / 16;
    for (int i = tid; i < 16 * KCH; i += NW * 32) {
      const int row = i / KCH, ch = i % KCH;
      bool valid;
      size_t ri;
      tok_ptr(t * 16 + row, valid, ri);
      const __nv_bfloat16* src = kbase + ri * DK + ch * 8;
      cp_async16(dst + row * KRS + ch * 16, valid ? (const void*)src : (const void*)kbase, valid ? 16 : 0);
    }
    cp_async_commit();
  };

  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  float oacc[kDVC / 8][4];
#pragma unroll
  for (int i = 0; i < kDVC / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  const float sl2 = d.scale * kLog2e;
  const int vcol0 = qq * kDVC;
  float* my_red = red + (ht * 4 + qq) * 256 + lane;     // fragment value j of the lane at [j * 32]

  auto process_tile = [&](int t, const unsigned char* kt) {
    float sacc[2][4];
#pragma unroll
    for (int nn = 0; nn < 2; ++nn) sacc[nn][0] = sacc[nn][1] = sacc[nn][2] = sacc[nn][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < QDIMS / 16; ++ks) {
      uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
      const int kc = qq * QDIMS + ks * 16;
      ldmatrix_x4(a0, a1, a2, a3, qs + (ht * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * KRS + (kc + (lane >> 4) * 8) * 2);
      ldmatrix_x4(b0, b1, b2, b3, kt + ((lane & 7) + (lane >> 4) * 8) * KRS + (kc + ((lane >> 3) & 1) * 8) * 2);
      mma_bf16_16816(sacc[0], a0, a1, a2, a3, b0, b1);
      mma_bf16_16816(sacc[1], a0, a1, a2, a3, b2, b3);
    }
    // sum the head tile's four quarter products (fragment layouts are identical), fixed order
#pragma unroll
    for (int j = 0; j < 8; ++j) my_red[j * 32] = sacc[j >> 2][j & 3];
    named_barrier(1 + ht, 128);
    const float* tile_red = red + ht * 4 * 256 + lane;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      sacc[j >> 2][j & 3] =
          ((tile_red[j * 32] + tile_red[256 + j * 32]) + tile_red[512 + j * 32]) + tile_red[768 + j * 32];
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int nn = 0; nn < 2; ++nn) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        bool valid;
        size_t ri;
        tok_ptr(t * 16 + nn * 8 + (lane & 3) * 2 + e, valid, ri);
        const float s_lo = valid ? sacc[nn][e] * sl2 : -INFINITY;
        const float s_hi = valid ? sacc[nn][2 + e] * sl2 : -INFINITY;
        sacc[nn][e] = s_lo;
        sacc[nn][2 + e] = s_hi;
        mx_lo = fmaxf(mx_lo, s_lo);
        mx_hi = fmaxf(mx_hi, s_hi);
      }
    }
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float al_lo = mn_lo == -INFINITY ? 1.f : exp2f(m_lo - mn_lo);
    const float al_hi = mn_hi == -INFINITY ? 1.f : exp2f(m_hi - mn_hi);
    float ps_lo = 0.f, ps_hi = 0.f;
#pragma unroll
    for (int nn = 0; nn < 2; ++nn) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float p_lo = mn_lo == -INFINITY ? 0.f : exp2f(sacc[nn][e] - mn_lo);
        const float p_hi = mn_hi == -INFINITY ? 0.f : exp2f(sacc[nn][2 + e] - mn_hi);
        sacc[nn][e] = p_lo;
        sacc[nn][2 + e] = p_hi;
        ps_lo += p_lo;
        ps_hi += p_hi;
      }
    }
    ps_lo += __shfl_xor_sync(0xffffffffu, ps_lo, 1);
    ps_lo += __shfl_xor_sync(0xffffffffu, ps_lo, 2);
    ps_hi += __shfl_xor_sync(0xffffffffu, ps_hi, 1);
    ps_hi += __shfl_xor_sync(0xffffffffu, ps_hi, 2);
    l_lo = l_lo * al_lo + ps_lo;
    l_hi = l_hi * al_hi + ps_hi;
    m_lo = mn_lo;
    m_hi = mn_hi;
    uint32_t ph[4], pl[4];
    auto split2 = [](float a, float b, uint32_t& hi, uint32_t& lo) {
      hi = pack_bf16x2(a, b);
      lo = pack_bf16x2(a - bf16_lo(hi), b - bf16_hi(hi));
    };
    split2(sacc[0][0], sacc[0][1], ph[0], pl[0]);
    split2(sacc[0][2], sacc[0][3], ph[1], pl[1]);
    split2(sacc[1][0], sacc[1][1], ph[2], pl[2]);
    split2(sacc[1][2], sacc[1][3], ph[3], pl[3]);
#pragma unroll
    for (int nd = 0; nd < kDVC / 8; nd += 2) {
      oacc[nd][0] *= al_lo; oacc[nd][1] *= al_lo; oacc[nd][2] *= al_hi; oacc[nd][3] *= al_hi;
      oacc[nd + 1][0] *= al_lo; oacc[nd + 1][1] *= al_lo; oacc[nd + 1][2] *= al_hi; oacc[nd + 1][3] *= al_hi;
      uint32_t b0, b1, b2, b3;
      const int trow = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int col = vcol0 + nd * 8 + (lane >> 4) * 8;
      ldmatrix_x4_trans(b0, b1, b2, b3, kt + trow * KRS + col * 2);
      mma_bf16_16816(oacc[nd], ph[0], ph[1], ph[2], ph[3], b0, b1);
      mma_bf16_16816(oacc[nd], pl[0], pl[1], pl[2], pl[3], b0, b1);
      mma_bf16_16816(oacc[nd + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
      mma_bf16_16816(oacc[nd + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
    }
  };

  int stage = 0;
  if (n_tiles > 0) load_tile(0, bufs);
  for (int t = 0; t < n_tiles; ++t, stage ^= 1) {
    if (t + 1 < n_tiles) {
      load_tile(t + 1, bufs + (stage ^ 1) * TILE);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    process_tile(t, bufs + stage * TILE);
    __syncthreads();        // the buffer and the score-reduction tiles are reused next
  }

  const int row_lo = ht * 16 + (lane >> 2), row_hi = row_lo + 8;     // within the CTA's 32 heads
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int row = hg * HEADS + (hh ? row_hi : row_lo);              // within the group of G
    const float m = hh ? m_hi : m_lo, l = hh ? l_hi : l_lo;
#pragma unroll
    for (int nd = 0; nd < kDVC / 8; ++nd) {
      const int c = vcol0 + nd * 8 + (lane & 3) * 2;
      const float o0 = oacc[nd][hh * 2], o1 = oacc[nd][hh * 2 + 1];
      if (n_split == 1) {
        float* dst = out + ((size_t)r * d.Hq + h * d.G + row) * d.dv + c;
        dst[0] = l > 0.f ? o0 / l : 0.f;
        dst[1] = l > 0.f ? o1 / l : 0.f;
      } else {
        float* dst = L.attn_part + (((size_t)u * n_split + split) * d.G + row) * d.dv + c;
        dst[0] = o0;
        dst[1] = o1;
      }
    }
    if (n_split > 1 && qq == 0 && (lane & 3) == 0) {
      L.attn_ml[(((size_t)u * n_split + split) * d.G + row) * 2 + 0] = m;
      L.attn_ml[(((size_t)u * n_split + split) * d.G + row) * 2 + 1] = l;
    }
  }
}

// out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s over the splits of a (unit, q head).
__global__ void __launch_bounds__(128) attn_combine_kernel(Dims d, Layer L, float* __restrict__ out, int n_split) {
  kvs_pdl_entry();
  const int u = blockIdx.x, g = blockIdx.y;
  const int r = u / d.Hkv, h = u % d.Hkv;
  const float* pml = L.attn_ml + ((size_t)u * n_split * d.G) * 2;
  float M = -INFINITY;
  for (int s = 0; s < n_split; ++s) M = fmaxf(M, pml[((size_t)s * d.G + g) * 2]);
  float lsum = 0.f;
  for (int s = 0; s < n_split; ++s) {
    float ms = pml[((size_t)s * d.G + g) * 2];
    if (ms != -INFINITY) lsum += exp2f(ms - M) * pml[((size_t)s * d.G + g) * 2 + 1];
  }
  for (int c = threadIdx.x; c < d.dv; c += blockDim.x) {
    float o = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < n_split; ++s) {
        float ms = pml[((size_t)s * d.G + g) * 2];
        if (ms != -INFINITY) o += exp2f(ms - M) * L.attn_part[(((size_t)u * n_split + s) * d.G + g) * d.dv + c];
      }
    }
    out[((size_t)r * d.Hq + h * d.G + g) * d.dv + c] = lsum > 0.f ? o / lsum : 0.f;
  }
}

}  // namespace
int attention_split(const Dims& d, int* n_split_out, int* bps_out);
namespace {

template <int DK, int MT, bool VSHARE>
cudaError_t launch_attn_t(const Dims& d, const Layer& L, const __nv_bfloat16* q, const int* sel,
                          const int* slot_of_sel, const int* nsel, const int* ctx_len, float* out, cudaStream_t s) {
  using Cfg = AttnCfg<DK, MT, VSHARE>;
  auto kern = attn_kernel<DK, MT, VSHARE>;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), Cfg::SMEM);
  if (e != cudaSuccess) return e;
  const int nz = d.dv / kDVC;
  int n_split, bps;
  if (!attention_split(d, &n_split, &bps)) return cudaErrorInvalidValue;
  dim3 grid(n_split, d.U, nz);
  launch_pdl(kern, dim3(grid), dim3(Cfg::NW * 32), Cfg::SMEM, s, d, L, q, sel, slot_of_sel, nsel, ctx_len, out, n_split, bps);
  e = cudaGetLastError();
  if (e != cudaSuccess || n_split == 1) return e;
  launch_pdl(attn_combine_kernel, dim3(dim3(d.U, d.G)), dim3(128), 0, s, d, L, out, n_split);
  return cudaGetLastError();
}

bool mla_path(const Dims& d) { return d.v_shares_k && d.dk == 576 && d.dv == 512 && d.G % mla::HEADS == 0; }

cudaError_t launch_attn_mla(const Dims& d, const Layer& L, const __nv_bfloat16* q, const int* sel,
                            const int* slot_of_sel, const int* nsel, const int* ctx_len, float* out, cudaStream_t s) {
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(attn_mla_kernel), mla::SMEM);
  if (e != cudaSuccess) return e;
  int n_split, bps;
  if (!attention_split(d, &n_split, &bps)) return cudaErrorInvalidValue;
  dim3 grid(n_split, d.U, d.G / mla::HEADS);
  launch_pdl(attn_mla_kernel, dim3(grid), dim3(mla::NW * 32), mla::SMEM, s, d, L, q, sel, slot_of_sel, nsel, ctx_len, out, n_split, bps);
  e = cudaGetLastError();
  if (e != cudaSuccess || n_split == 1) return e;
  launch_pdl(attn_combine_kernel, dim3(dim3(d.U, d.G)), dim3(128), 0, s, d, L, out, n_split);
  return cudaGetLastError();
}

}  // namespace

int attention_split(const Dims& d, int* n_split_out, int* bps_out) {
  // grid z: value chunks, or head groups on the MLA path
  const int nz = mla_path(d) ? d.G / mla::HEADS : d.dv / kDVC;
  // CTAs of the launched configuration that fit on one SM (shared memory bound)
  int smem = AttnCfg<128, 1, false>::SMEM;
  if (d.v_shares_k) smem = d.G <= 16 ? AttnCfg<576, 1, true>::SMEM : AttnCfg<576, 8, true>::SMEM;
  if (mla_path(d)) smem = mla::SMEM;
  const int per_sm = max(1, min(2, (227 * 1024) / (smem + 1024)));
  const int slots = device_sm_count() * per_sm;
  // split count with the least time: waves (rounded up) x (selection share of a CTA + a fixed
  // per-CTA cost, ~3% of a whole selection); at least 2 blocks per split
  const int cap = max(1, min(kAttnSplitMax, (d.Kb + 1) / 2));
  int n_split = 1;
  double best = 1e30;
  for (int n = 1; n <= cap; ++n) {
    const long long ctas = (long long)d.U * nz * n;
    const double cost = (double)((ctas + slots - 1) / slots) * (1.0 / n + 0.03);
    if (cost < best) {
      best = cost;
      n_split = n;
    }
  }
  int bps = (d.Kb + n_split - 1) / n_split;
  const int max_blocks_cta = 4 * 1024 / 8;
  if (bps > max_blocks_cta) {
    n_split = (d.Kb + max_blocks_cta - 1) / max_blocks_cta;
    if (n_split > kAttnSplitMax) return 0;
    bps = (d.Kb + n_split - 1) / n_split;
  }
  *n_split_out = (d.Kb + bps - 1) / bps;
  *bps_out = bps;
  return 1;
}

int attention_supported(const Dims& d) {
  if (d.fp8) return attention_tma_supported(d);   // E4M3 tiles: the TMA kernel only
  if (d.dv % kDVC) return 0;
  if (d.v_shares_k) return d.dk == 576 && d.dv <= 512 && (d.G <= 16 || (mla_path(d) && d.G <= 128) || d.G == 128);
  return d.dk == 128 && d.dv == 128 && d.G <= 16;
}

cudaError_t launch_attention(const Dims& d, const Layer& L, const __nv_bfloat16* q, const int* sel,
                             const int* slot_of_sel, const int* nsel, const int* ctx_len, float* out,
                             cudaStream_t s) {
  if (!attention_supported(d)) return cudaErrorInvalidValue;
  if (attention_tma_supported(d) && L.tmK && L.tmV)
    return launch_attention_tma(d, L, L.tmK, L.tmV, q, sel, slot_of_sel, nsel, ctx_len, out, s);
  if (d.fp8) return cudaErrorInvalidValue;
  if (d.v_shares_k) {
    if (d.G <= 16) return launch_attn_t<576, 1, true>(d, L, q, sel, slot_of_sel, nsel, ctx_len, out, s);
    if (attention_mla_tc_supported(d)) return launch_attention_mla_tc(d, L, q, sel, slot_of_sel, nsel, ctx_len, out, s);
    if (mla_path(d)) return launch_attn_mla(d, L, q, sel, slot_of_sel, nsel, ctx_len, out, s);
    return launch_attn_t<576, 8, true>(d, L, q, sel, slot_of_sel, nsel, ctx_len, out, s);
  }
  return launch_attn_t<128, 1, false>(d, L, q, sel, slot_of_sel, nsel, ctx_len, out, s);
}

}  // namespace kvs
