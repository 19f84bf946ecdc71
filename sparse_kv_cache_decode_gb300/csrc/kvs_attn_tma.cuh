// Decode attention over the selected cache slots (one CTA's work; shared by the attention kernel
// and the fused layer kernel), TMA-pipelined (GQA groups of up to 16 q heads,
// head dim 128, block size a multiple of 16).
//
// The (unit, selected block, 16-row sub-tile) sequence of a layer is cut into equal contiguous
// ranges, one per CTA, with exactly 2 CTAs per SM (room for a fetch CTA beside them).  In each
// CTA one producer thread streams the K and V tiles of its range into a shared-memory ring, one 2D
// tensor load per tile (the pool seen as 128-byte lines, 32 lines per 16-row tile, 128-byte
// swizzle; completion on an mbarrier per stage: few large loads, as each load has a fixed cost
// that dominates with small boxes); the consumer warps take the
// tiles round-robin, each keeping an online softmax per q head on tensor-core tiles with the
// tokens on the MMA's M side (a decode group has only a few heads, so the heads fill one or two
// n8 tiles instead of a mostly empty m16 tile):
//   S^T  = K (16 tokens x 128) . Q^T (128 x 8 heads)
//   O^T += V^T (128 x 16 tokens) . P^T (16 tokens x 8 heads), P split into bf16 high and low parts,
// with P^T's fragments made from S^T's by an 8x8 register transpose (movmatrix).
// At the end of a unit each consumer warp leaves its state in a shared-memory slot without waiting
// for the other warps (the stream of tiles goes on); when the CTA's range is done, the warps'
// states are combined into one partial (unnormalised O, max, sum) per head and unit, the CTA
// counts its partial of each unit it touched, and the last CTA of a unit to finish (a per-unit
// counter) merges the unit's partials: o = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p.
// The CTA's block ids, slots and the units' lengths are staged in shared memory first (one round
// of global loads), so the producer issues tensor loads without waiting on global memory.
// Every mbarrier wait is bounded by the context's wait timeout (KVS_ERR_TIMEOUT on expiry).
// E4M3 slot pools: a stage holds 16 rows x 128 codes of K and of V (one 16-row box each); the
// consumer warp widens its tile into a bf16 copy in the layout of a bf16 stage in its own staging
// area (every E4M3 value is exact in bf16), releases the stage, and runs the same tiles; the K
// scale joins the softmax scale and the V scale is applied at the merge.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>

#include "kvs_common.cuh"
#include "kvs_ptx.cuh"

namespace kvs {
namespace tma {

constexpr int D = 128;
constexpr int kStages = 8;
constexpr int kConsumers = 4;
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kCtasPerSm = 2;               // leaves registers for a fetch CTA beside them
constexpr int kTile = 16 * D * 2;           // bytes of a 16-row bf16 K or V tile
constexpr int kStage = 2 * kTile;
constexpr int kMaxPos = 1024;               // positions (selected blocks) per CTA
constexpr int kMaxUnits = 64;               // units one CTA's range may touch
constexpr int kMergeChunk = 16;            // partials the merge reads in one round of loads
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory of the kernel (offsets from a 1024-byte aligned base): the stage ring, per-warp
// bf16 staging (E4M3 pools only), barriers, flags, the units' lengths, counts and last-CTA flags,
// the consumer warps' combine slots (max and sum per head; O rows of the group's G heads), then
// the CTA's block and slot lists (per_cta entries each).
template <int NT, bool FP8>
struct Smem {
  static constexpr int kHeads = 8 * NT;                                  // head columns of the tiles
  static constexpr int kSlots = NT == 1 ? 2 : 1;                         // deferred combine slots
  static constexpr int kStageBytes = FP8 ? 2 * 16 * D : kStage;
  static constexpr int kRing = kStages * kStageBytes;
  static constexpr int kStaging = FP8 ? kConsumers * kStage : 0;
  static constexpr int kBars = kRing + kStaging;
  static constexpr int kFlags = kBars + 2 * kStages * 8;
  static constexpr int kUnits = kFlags + 64;                             // u_len, u_n, u_last_cta
  static constexpr int kCmbMl = kUnits + 3 * kMaxUnits * 4;              // [slot][warp][head][2]: max, sum
  static constexpr int kCmb = kCmbMl + kSlots * kConsumers * kHeads * 8; // [slot][warp][G][D] floats
  __host__ __device__ static int lists(int G) { return kCmb + kSlots * kConsumers * G * D * 4; }   // m_blk, m_slot
  static int bytes(int G, int per_cta) { return lists(G) + 2 * per_cta * 4 + 1024; }   // + alignment slack
};

// Two E4M3 codes (bits 0-7, 8-15) -> bf16x2, exactly (through f16, which holds every E4M3 value).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two));
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
  return pack_bf16x2(f.x, f.y);
}

// Byte offset of the 16-byte chunk holding (row, col) of a 16-row bf16 tile as one tensor load of
// 32 lines of 128 bytes writes it with the 128-byte swizzle: line = 2 row + col / 64, chunk index
// XOR (line % 8).
__device__ __forceinline__ int tile_off(int row, int col) {
  const int line = 2 * row + (col >> 6);
  return line * 128 + ((((col & 63) >> 3) ^ (line & 7)) << 4);
}

// Transpose of an 8x8 b16 matrix held one row pair per lane (lane l: row l/4, columns 2(l%4), +1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
  return d;
}

// phase: 0 every selected position, partials merged; 1 only the positions that hit in the last
// update (miss_flag 0), partials kept; 2 only the positions that missed, then the unit's partials
// of both phases merged.  Phases 1 and 2 use the same split (their partials side by side).
struct Plan {
  int n_cta, per_cta, max_segs, phase;
};

// The split of the layer's (unit, block) positions over `ctas` CTAs (fewer when the caps bind).
__host__ __device__ inline Plan make_plan_ctas(const Dims& d, int ctas) {
  Plan p;
  const long long positions = (long long)d.U * d.Kb;
  if (ctas < 1) ctas = 1;
  p.per_cta = (int)((positions + ctas - 1) / ctas);
  // at most 256 partials (segments) per unit (bounds the workspace's partial slots)
  const int seg_cap = 255;
  const int min_per = (d.Kb + seg_cap - 1) / seg_cap;
  if (p.per_cta < min_per) p.per_cta = min_per;
  if (p.per_cta < 1) p.per_cta = 1;
  if (p.per_cta > kMaxPos) p.per_cta = kMaxPos;
  if ((long long)p.per_cta > (long long)(kMaxUnits - 2) * d.Kb) p.per_cta = (kMaxUnits - 2) * d.Kb;
  p.n_cta = (int)((positions + p.per_cta - 1) / p.per_cta);
  p.max_segs = (d.Kb + p.per_cta - 1) / p.per_cta + 1;
  p.phase = 0;
  return p;
}

__host__ __device__ inline Plan make_plan(const Dims& d, int n_sm) { return make_plan_ctas(d, n_sm * kCtasPerSm); }

__device__ __forceinline__ int rows_present(int len, int blk, int bs) { return min(bs, len - blk * bs); }

// Attention CTA c of the plan (every thread of a kThreads-thread CTA calls it); tmK / tmV must be
// kernel parameters (grid constants) of the calling kernel.
template <int NT, bool FP8>  // NT: n8 tiles of q heads (G <= 8: 1, G <= 16: 2)
__device__ __forceinline__ void attn_tma_cta(const CUtensorMap& tmK, const CUtensorMap& tmV, const Dims& d,
                                             const Layer& L, const __nv_bfloat16* __restrict__ q,
                                             const int* __restrict__ sel, const int* __restrict__ slot_of_sel,
                                             const int* __restrict__ nsel, const int* __restrict__ ctx_len,
                                             float* __restrict__ out, const Plan& plan, int c,
                                             unsigned char* smem_raw) {
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using Lay = Smem<NT, FP8>;
  constexpr int H8 = Lay::kHeads;
  constexpr int kSlots = Lay::kSlots;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBars);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kFlags);
  int* u_len = reinterpret_cast<int*>(smem + Lay::kUnits);       // [kMaxUnits]
  int* u_n = u_len + kMaxUnits;                                  // [kMaxUnits]
  int* u_last_cta = u_n + kMaxUnits;                             // [kMaxUnits]: this CTA merges the unit
  int* m_blk = reinterpret_cast<int*>(smem + Lay::lists(d.G));   // [per_cta], -1: none
  int* m_slot = m_blk + plan.per_cta;                            // [per_cta]
  float* cmb = reinterpret_cast<float*>(smem + Lay::kCmb);       // [slot][warp][G][D]
  float* cmb_ml = reinterpret_cast<float*>(smem + Lay::kCmbMl);  // [slot][warp][H8][2]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kConsumers && lane == 0) {   // the maps are kernel parameters, not outputs of earlier kernels
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  kvs_pdl_entry();   // every global memory access below follows the wait

  const long long p0 = (long long)c * plan.per_cta;
  const long long p1 = min((long long)d.U * d.Kb, p0 + plan.per_cta);
  const int subs = d.bs / 16;
  const uint64_t timeout_ns = (uint64_t)d.timeout_us * 1000ull;
  const int u_first = (int)(p0 / d.Kb), u_last = (int)((p1 - 1) / d.Kb);

  // one round of global loads: the units' lengths and counts, the range's (block, slot) pairs
  for (int j = tid; j <= u_last - u_first; j += blockDim.x) {
    u_len[j] = ctx_len[(u_first + j) / d.Hkv];
    u_n[j] = nsel[u_first + j];
  }
  constexpr int kOtherPhase = -0x40000000;   // a position of the other phase: skipped, no error
  for (int i = tid; i < (int)(p1 - p0); i += blockDim.x) {
    int b = sel[p0 + i];
    if (plan.phase != 0 && ((plan.phase == 1) == (L.miss_flag[p0 + i] != 0))) b = kOtherPhase;
    m_blk[i] = b;
    m_slot[i] = slot_of_sel[p0 + i];
  }
  __syncthreads();
  // validate in shared memory: an out-of-range length, count, block id or slot is reported as
  // KVS_ERR_BAD_INDEX and its tiles are skipped (no tensor load ever addresses another unit's slots)
  for (int i = tid; i < (int)(p1 - p0); i += blockDim.x) {
    const long long p = p0 + i;
    const int uj = (int)(p / d.Kb) - u_first, ii = (int)(p % d.Kb);
    const int len = u_len[uj], n = u_n[uj];
    const bool unit_ok = len >= 0 && len <= d.max_ctx && n >= 0 && n <= d.Kb;
    if (!unit_ok && ii == 0) set_error(L.err, KVS_ERR_BAD_INDEX);
    int blk = -1;
    if (unit_ok && ii < n && m_blk[i] != kOtherPhase) {
      blk = m_blk[i];
      const int slot = m_slot[i];
      if (blk < 0 || blk >= n_blocks_of(len, d.bs) || slot < 0 || slot >= d.C) {
        set_error(L.err, KVS_ERR_BAD_INDEX);
        blk = -1;
      }
    }
    m_blk[i] = blk;
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ------------------------------------------------------------------ producer
    if (lane != 0) return;
    int k = 0;
    bool ok = true;
    for (long long p = p0; p < p1 && ok; ++p) {
      const int u = (int)(p / d.Kb);
      const int blk = m_blk[p - p0], slot = m_slot[p - p0];
      if (blk < 0) continue;
      const int rows = rows_present(u_len[u - u_first], blk, d.bs);
      for (int sub = 0; sub < subs && ok; ++sub) {
        if (sub * 16 >= rows) break;
        const int s = k % kStages;
        if (k >= kStages && !mbar_wait(&empty[s], ((k / kStages) & 1) ^ 1, timeout_ns)) {
          ok = false;
          break;
        }
        if (*abort_flag) { ok = false; break; }
        const int y = ((u * d.C + slot) * d.bs) + sub * 16;
        unsigned char* st = smem + s * Lay::kStageBytes;
        mbar_arrive_expect_tx(&full[s], Lay::kStageBytes);
        if (FP8) {
          tma_load_2d(st, &tmK, 0, y, &full[s]);
          tma_load_2d(st + 16 * 128, &tmV, 0, y, &full[s]);
        } else {   // one 32-line box per tile: the pools seen as 128-byte lines (two per row)
          tma_load_2d(st, &tmK, 0, 2 * y, &full[s]);
          tma_load_2d(st + kTile, &tmV, 0, 2 * y, &full[s]);
        }
        ++k;
      }
    }
    if (!ok) {
      set_error(L.err, KVS_ERR_TIMEOUT);
      *abort_flag = 1;
    }
    // do not leave while tensor loads into this CTA's shared memory may be in flight; this wait has
    // its own fixed bound, so a short caller timeout cannot retire the CTA under a pending load
    for (int j = max(0, k - kStages); j < k; ++j) mbar_wait(&full[j % kStages], (j / kStages) & 1, kDrainTimeoutNs);
    return;
  }

  // -------------------------------------------------------------------- consumers
  const int G = d.G;
  const float sl2 = FP8 ? d.scale * d.k_scale * kLog2e : d.scale * kLog2e;
  const int tq = lane >> 2, hq = (lane & 3) * 2;   // fragment row (token or dim) and head column pair
  int k = 0;          // position in the CTA's tile sequence
  bool ok = true;
  const int n_imm = max(0, u_last - u_first + 1 - kSlots);   // units combined at their end
  // the CTA's partial of unit u from the consumer warps' states in combine slot `slot`, merged in
  // warp order: O = sum_w 2^(m_w - M) O_w, l = sum_w 2^(m_w - M) l_w, M = max_w m_w
  auto combine = [&](int u, int slot) {
    const int c0 = (int)(((long long)u * d.Kb) / plan.per_cta);
    const size_t pidx = (size_t)u * plan.max_segs * (plan.phase ? 2 : 1) + (plan.phase == 2 ? plan.max_segs : 0) +
                        (size_t)(c - c0);
    const float* sw = cmb + slot * kConsumers * G * D;
    const float* sml = cmb_ml + slot * kConsumers * H8 * 2;
    for (int e = tid; e < G * (D / 4); e += kConsumers * 32) {
      const int g = e / (D / 4), c4 = e % (D / 4);
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, sml[(w * H8 + g) * 2]);
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      float lsum = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        const float mw = sml[(w * H8 + g) * 2];
        const float wgt = (M == -INFINITY || mw == -INFINITY) ? 0.f : exp2f(mw - M);
        const float4 x = reinterpret_cast<const float4*>(sw + (w * G + g) * D)[c4];
        o.x += wgt * x.x;
        o.y += wgt * x.y;
        o.z += wgt * x.z;
        o.w += wgt * x.w;
        lsum += wgt * sml[(w * H8 + g) * 2 + 1];
      }
      reinterpret_cast<float4*>(L.attn_part + (pidx * G + g) * D)[c4] = o;
      if (c4 == 0) *reinterpret_cast<float2*>(L.attn_ml + (pidx * G + g) * 2) = make_float2(M, lsum);
    }
  };
  for (int u = u_first; u <= u_last; ++u) {
    const int r = u / d.Hkv, h = u % d.Hkv;
    const int len = u_len[u - u_first];
    // Q^T as m16n8k16 B fragments: head tq of each n8 tile, dims 2(lane%4), +1 and those + 8
    uint32_t qb[D / 16][NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int g = nt * 8 + tq;
      const uint32_t* qr = reinterpret_cast<const uint32_t*>(q + ((size_t)r * d.Hq + h * G + min(g, G - 1)) * D);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qb[ks][nt][0] = g < G ? qr[(ks * 16 + hq) >> 1] : 0u;
        qb[ks][nt][1] = g < G ? qr[(ks * 16 + 8 + hq) >> 1] : 0u;
      }
    }
    // per head column (hq + j of each n8 tile): the running max, uniform over the 8 lanes of the
    // column, and this lane's share of the running sum (reduced over those lanes at the unit's end)
    float m_run[NT][2], l_run[NT][2];
    float oacc[D / 16][NT][4];   // O^T: dims mt*16 + tq (and + 8) x heads hq, hq + 1
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt][0] = m_run[nt][1] = -INFINITY;
      l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) oacc[mt][nt][0] = oacc[mt][nt][1] = oacc[mt][nt][2] = oacc[mt][nt][3] = 0.f;
    }

    const long long pu0 = max(p0, (long long)u * d.Kb), pu1 = min(p1, (long long)(u + 1) * d.Kb);
    for (long long p = pu0; p < pu1; ++p) {
      const int blk = m_blk[p - p0];
      if (blk < 0) continue;
      const int rows = rows_present(len, blk, d.bs);
      for (int sub = 0; sub < subs; ++sub) {
        if (sub * 16 >= rows) break;
        const int kk = k++;
        if ((kk % kConsumers) != warp || !ok) continue;
        const int s = kk % kStages;
        if (!mbar_wait(&full[s], (kk / kStages) & 1, timeout_ns)) {
          // give up on the remaining tiles, but still write and count this unit's partials below,
          // so that the per-unit completion counters stay consistent for later launches
          ok = false;
          *abort_flag = 1;
          continue;
        }
        const unsigned char* kt = smem + s * kStage;
        if (FP8) {
          // widen the stage's K and V codes into this warp's bf16 staging (the layout of a bf16
          // stage), then release the stage
          unsigned char* stg = smem + Lay::kRing + warp * kStage;
          const unsigned char* src = smem + s * Lay::kStageBytes;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int qi = lane + 32 * j;
            const int tile = qi >> 7, row = (qi >> 3) & 15, c16 = qi & 7;
            const uint4 v = *reinterpret_cast<const uint4*>(src + tile * 2048 + row * 128 + ((c16 ^ (row & 7)) << 4));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              o[2 * e] = e4m3x2_to_bf16x2(w[e] & 0xffffu);
              o[2 * e + 1] = e4m3x2_to_bf16x2(w[e] >> 16);
            }
            unsigned char* dst = stg + tile * kTile;
            *reinterpret_cast<uint4*>(dst + tile_off(row, c16 * 16)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(dst + tile_off(row, c16 * 16 + 8)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
          kt = stg;
        }
        const unsigned char* vt = kt + kTile;
        const int valid_rows = rows - sub * 16;     // tokens of this tile before the context end
        // S^T = K Q^T in two accumulator chains (even and odd 16-dim chunks) per n8 tile
        float sacc[NT][2][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) sacc[nt][ch][0] = sacc[nt][ch][1] = sacc[nt][ch][2] = sacc[nt][ch][3] = 0.f;
        {
          // A fragments of K: 8x8 matrices (t 0-7, d 0-7), (t 8-15, d 0-7), (t 0-7, d 8-15), (t 8-15, d 8-15)
          const int trow = (lane & 7) + ((lane >> 3) & 1) * 8;
          const int dcol = (lane >> 4) * 8;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(a0, a1, a2, a3, kt + tile_off(trow, ks * 16 + dcol));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(sacc[nt][ks & 1], a0, a1, a2, a3, qb[ks][nt][0], qb[ks][nt][1]);
          }
        }
        // online softmax per head column in the log2 domain; tokens past the context end are masked
        uint32_t pb[NT][4];   // P^T B fragments: high part (t 0-7, t 8-15), low part (t 0-7, t 8-15)
        float alpha[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float sv[4];   // (t = tq, head hq), (tq, hq + 1), (tq + 8, hq), (tq + 8, hq + 1)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = tq + (e >> 1) * 8;
            sv[e] = tok < valid_rows ? (sacc[nt][0][e] + sacc[nt][1][e]) * sl2 : -INFINITY;
          }
          float pv[4];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(sv[j], sv[2 + j]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m_run[nt][j], mx);
            alpha[nt][j] = mn == -INFINITY ? 1.f : exp2f(m_run[nt][j] - mn);
            pv[j] = mn == -INFINITY ? 0.f : exp2f(sv[j] - mn);
            pv[2 + j] = mn == -INFINITY ? 0.f : exp2f(sv[2 + j] - mn);
            l_run[nt][j] = l_run[nt][j] * alpha[nt][j] + pv[j] + pv[2 + j];
            m_run[nt][j] = mn;
          }
          const uint32_t h0 = pack_bf16x2(pv[0], pv[1]), h1 = pack_bf16x2(pv[2], pv[3]);
          const uint32_t l0 = pack_bf16x2(pv[0] - bf16_lo(h0), pv[1] - bf16_hi(h0));
          const uint32_t l1 = pack_bf16x2(pv[2] - bf16_lo(h1), pv[3] - bf16_hi(h1));
          pb[nt][0] = movmatrix_trans(h0);
          pb[nt][1] = movmatrix_trans(h1);
          pb[nt][2] = movmatrix_trans(l0);
          pb[nt][3] = movmatrix_trans(l1);
        }
        // O^T = alpha O^T + V^T P^T; A fragments of V^T by transposing loads of the token rows:
        // 8x8 matrices (d 0-7, t 0-7), (d 8-15, t 0-7), (d 0-7, t 8-15), (d 8-15, t 8-15)
        {
          const int trow = (lane & 7) + (lane >> 4) * 8;
          const int dcol = ((lane >> 3) & 1) * 8;
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4_trans(a0, a1, a2, a3, vt + tile_off(trow, mt * 16 + dcol));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              oacc[mt][nt][0] *= alpha[nt][0];
              oacc[mt][nt][1] *= alpha[nt][1];
              oacc[mt][nt][2] *= alpha[nt][0];
              oacc[mt][nt][3] *= alpha[nt][1];
              mma_bf16_16816(oacc[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
              mma_bf16_16816(oacc[mt][nt], a0, a1, a2, a3, pb[nt][2], pb[nt][3]);
            }
          }
        }
        __syncwarp();
        if (!FP8 && lane == 0) mbar_arrive(&empty[s]);
      }
    }
    // this warp's state of unit u goes to a combine slot in shared memory: the CTA's last kSlots
    // units each keep a slot until the CTA's range is done; earlier units (ranges of more units
    // than slots) are combined at once, behind a barrier, in slot 0
    const int j = u - u_first;
    const int slot = j < n_imm ? 0 : j - n_imm;
    float* tw = cmb + (slot * kConsumers + warp) * G * D;
    float* tml = cmb_ml + (slot * kConsumers + warp) * H8 * 2;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        float lsum = l_run[nt][jj];
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 4);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 8);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);
        const int g = nt * 8 + hq + jj;
        if (tq == 0) {
          tml[g * 2 + 0] = m_run[nt][jj];
          tml[g * 2 + 1] = lsum;
        }
        if (g < G) {
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            tw[g * D + mt * 16 + tq] = oacc[mt][nt][jj];
            tw[g * D + mt * 16 + 8 + tq] = oacc[mt][nt][2 + jj];
          }
        }
      }
    if (j < n_imm) {
      named_bar_sync(1, kConsumers * 32);
      combine(u, 0);
      named_bar_sync(1, kConsumers * 32);
    }
  }
  // combine the deferred units; then count this CTA's partial of each unit it touched (one thread
  // per unit); the last CTA of a unit to finish merges the unit's partials:
  // o = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p, in ascending order, one warp per q head,
  // 4 columns per lane.  The counter goes back to 0 for the next launch.
  named_bar_sync(1, kConsumers * 32);
  for (int u = u_first + n_imm; u <= u_last; ++u) combine(u, u - u_first - n_imm);
  if (plan.phase == 1) {   // the partials wait for the second phase's merge
    if (!ok) set_error(L.err, KVS_ERR_TIMEOUT);
    return;
  }
  __threadfence();
  named_bar_sync(1, kConsumers * 32);
  for (int j = tid; j <= u_last - u_first; j += kConsumers * 32) {
    const int u = u_first + j;
    const int c0 = (int)(((long long)u * d.Kb) / plan.per_cta);
    const int c1 = min(plan.n_cta - 1, (int)(((long long)(u + 1) * d.Kb - 1) / plan.per_cta));
    u_last_cta[j] = atomicAdd(&L.unit_done[u], 1u) == (unsigned)(c1 - c0);
  }
  named_bar_sync(1, kConsumers * 32);
  bool merged = false;
  for (int u = u_first; u <= u_last; ++u) {
    if (!u_last_cta[u - u_first]) continue;
    if (!merged) __threadfence();
    merged = true;
    const int c0 = (int)(((long long)u * d.Kb) / plan.per_cta);
    const int c1 = min(plan.n_cta - 1, (int)(((long long)(u + 1) * d.Kb - 1) / plan.per_cta));
    const int np = c1 - c0 + 1;
    const size_t base = (size_t)u * plan.max_segs * (plan.phase ? 2 : 1);
    const int np_all = plan.phase == 2 ? 2 * np : np;   // with the first phase's partials
    auto pix = [&](int p) { return base + (size_t)(p < np ? p : plan.max_segs + (p - np)); };
    const int r_out = u / d.Hkv, h_out = u % d.Hkv;
    for (int g = warp; g < G; g += kConsumers) {
      // chunks of kMergeChunk partials, each read in one round of loads (the (max, sum) pairs and the rows
      // together), merged online: the running state is rescaled when a chunk raises the max
      float M = -INFINITY, lpart = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q0 = 0; q0 < np_all; q0 += kMergeChunk) {
        const int nj = min(kMergeChunk, np_all - q0);
        float2 ml = make_float2(-INFINITY, 0.f);
        if (lane < nj) ml = __ldcg(reinterpret_cast<const float2*>(L.attn_ml + (pix(q0 + lane) * G + g) * 2));
        float4 x[kMergeChunk];
#pragma unroll
        for (int kq = 0; kq < kMergeChunk; ++kq)
          x[kq] = kq < nj ? __ldcg(reinterpret_cast<const float4*>(L.attn_part + (pix(q0 + kq) * G + g) * D) + lane)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        float mc = ml.x;
#pragma unroll
        for (int o = 16; o; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
        const float Mn = fmaxf(M, mc);
        const float a = (M == -INFINITY) ? 0.f : exp2f(M - Mn);   // rescale of the running state
        acc.x *= a; acc.y *= a; acc.z *= a; acc.w *= a;
        lpart *= a;
        const float wgt = (Mn == -INFINITY || ml.x == -INFINITY) ? 0.f : exp2f(ml.x - Mn);
        lpart += wgt * ml.y;   // this lane's share; summed over the lanes below
#pragma unroll
        for (int kq = 0; kq < kMergeChunk; ++kq) {
          const float wj = __shfl_sync(0xffffffffu, wgt, kq);
          acc.x += wj * x[kq].x;
          acc.y += wj * x[kq].y;
          acc.z += wj * x[kq].z;
          acc.w += wj * x[kq].w;
        }
        M = Mn;
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) lpart += __shfl_xor_sync(0xffffffffu, lpart, o);
      const float inv = lpart > 0.f ? (FP8 ? d.v_scale / lpart : 1.f / lpart) : 0.f;
      float4 res = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      reinterpret_cast<float4*>(out + ((size_t)r_out * d.Hq + h_out * G + g) * d.dv)[lane] = res;
    }
    if (tid == 0) L.unit_done[u] = 0u;
  }
  if (!ok) set_error(L.err, KVS_ERR_TIMEOUT);
}

}  // namespace tma
}  // namespace kvs
