// Decode attention over the selected cache slots, TMA-pipelined (GQA groups of up to 16 q heads,
// head dim 128, block size a multiple of 16).
//
// The (unit, selected block, 16-row sub-tile) sequence of a layer is cut into equal contiguous
// ranges, one per CTA, with exactly 2 CTAs per SM (room for a fetch CTA beside them).  In each
// CTA one producer thread streams the K and V tiles of its range into an 8-stage shared-memory ring with 2D tensor loads (128-byte
// swizzle, completion on an mbarrier per stage); 4 consumer warps take the tiles round-robin,
// each keeping an online softmax per q head on tensor-core tiles:
//   S  = Q (16 heads x 128) . K^T (128 x 16 tokens)
//   O += P (16 x 16) . V (16 x 128), P split into bf16 high and low parts.
// A warp writes its (unnormalised O, max, sum) for every unit its CTA touches; the last CTA of a
// unit to finish (a per-unit counter) merges that unit's partials:
// o = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p.
// The CTA's block ids, slots and the units' lengths are staged in shared memory first, so the
// producer issues tensor loads without waiting on global memory.
// Every mbarrier wait is bounded by the context's wait timeout (KVS_ERR_TIMEOUT on expiry).
// E4M3 slot pools: a stage holds 16 rows x 128 codes of K and of V (one 128-byte box each); the
// consumer warp widens its tile into a bf16 copy of the same swizzled layout in its own staging
// area (every E4M3 value is exact in bf16), releases the stage, and runs the same tiles; the K
// scale joins the softmax scale and the V scale is applied at the merge.
#include <cuda.h>
#include <cuda_fp16.h>

#include "kvs_common.cuh"
#include "kvs_ptx.cuh"

namespace kvs {

namespace {

constexpr int D = 128;
constexpr int kStages = 8;
constexpr int kConsumers = 4;
constexpr int kCtasPerSm = 2;   // leaves registers for a fetch CTA beside them
constexpr int kTile = 16 * D * 2;           // bytes of a 16-row K or V tile (two 64-column boxes)
constexpr int kStage = 2 * kTile;
constexpr int kMaxPos = 1024;               // positions (selected blocks) per CTA
constexpr int kMaxUnits = 64;               // units one CTA's range may touch
// Shared memory of the kernel: the stage ring, per-warp bf16 staging (E4M3 pools only), barriers,
// flags and the CTA's block and slot lists.
template <bool FP8>
struct Smem {
  static constexpr int kStageBytes = FP8 ? 2 * 16 * D : kStage;
  static constexpr int kRing = kStages * kStageBytes;
  static constexpr int kStaging = FP8 ? kConsumers * kStage : 0;
  static constexpr int kBars = kRing + kStaging;
  static constexpr int kTotal = kBars + 1024 + 2 * kStages * 8 + 64 + kMaxPos * 8 + kMaxUnits * 8;
};

// Two E4M3 codes (bits 0-7, 8-15) -> bf16x2, exactly (through f16, which holds every E4M3 value).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two));
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
  return pack_bf16x2(f.x, f.y);
}
constexpr float kLog2e = 1.4426950408889634f;

struct Plan {
  int n_cta, per_cta, max_segs;
};

__host__ __device__ inline Plan make_plan(const Dims& d, int n_sm) {
  Plan p;
  const long long positions = (long long)d.U * d.Kb;
  int ctas = n_sm * kCtasPerSm;
  p.per_cta = (int)((positions + ctas - 1) / ctas);
  // at most 1024 partials (segments x warps) per unit (bounds the workspace's partial slots)
  const int seg_cap = 1024 / kConsumers - 1;
  const int min_per = (d.Kb + seg_cap - 1) / seg_cap;
  if (p.per_cta < min_per) p.per_cta = min_per;
  if (p.per_cta < 1) p.per_cta = 1;
  if (p.per_cta > kMaxPos) p.per_cta = kMaxPos;
  if ((long long)p.per_cta > (long long)(kMaxUnits - 2) * d.Kb) p.per_cta = (kMaxUnits - 2) * d.Kb;
  p.n_cta = (int)((positions + p.per_cta - 1) / p.per_cta);
  p.max_segs = (d.Kb + p.per_cta - 1) / p.per_cta + 1;
  return p;
}

__device__ __forceinline__ int rows_present(int len, int blk, int bs) { return min(bs, len - blk * bs); }

template <bool ROWS8, bool FP8>  // ROWS8: G <= 8, fragment rows 8..15 are zero at compile time
__global__ void __launch_bounds__((kConsumers + 1) * 32, kCtasPerSm)
    attn_tma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, Dims d,
                    Layer L, const __nv_bfloat16* __restrict__ q, const int* __restrict__ sel,
                    const int* __restrict__ slot_of_sel, const int* __restrict__ nsel,
                    const int* __restrict__ ctx_len, float* __restrict__ out, Plan plan) {
  kvs_pdl_entry();
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using Lay = Smem<FP8>;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBars);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);
  volatile int* last_flag = abort_flag + 1;   // this CTA finished a unit last (consumers)
  int* m_blk = reinterpret_cast<int*>(smem + Lay::kBars + 2 * kStages * 8 + 64);       // [kMaxPos], -1: none
  int* m_slot = m_blk + kMaxPos;                                                       // [kMaxPos]
  int* u_len = m_slot + kMaxPos;                                                       // [kMaxUnits]
  int* u_n = u_len + kMaxUnits;                                                        // [kMaxUnits]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  const long long p0 = (long long)c * plan.per_cta;
  const long long p1 = min((long long)d.U * d.Kb, p0 + plan.per_cta);
  const int subs = d.bs / 16;
  const uint64_t timeout_ns = (uint64_t)d.timeout_us * 1000ull;

  const int u_first = (int)(p0 / d.Kb), u_last = (int)((p1 - 1) / d.Kb);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  // stage the units' lengths and the range's (block, slot) pairs; an out-of-range length, count,
  // block id or slot is reported as KVS_ERR_BAD_INDEX and its tiles are skipped (no tensor load
  // ever addresses another unit's slots)
  for (int j = tid; j <= u_last - u_first; j += blockDim.x) {
    int len = ctx_len[(u_first + j) / d.Hkv];
    int n = nsel[u_first + j];
    if (len < 0 || len > d.max_ctx || n < 0 || n > d.Kb) {
      set_error(L.err, KVS_ERR_BAD_INDEX);
      len = 0;
      n = 0;
    }
    u_len[j] = len;
    u_n[j] = n;
  }
  __syncthreads();
  for (int i = tid; i < (int)(p1 - p0); i += blockDim.x) {
    const long long p = p0 + i;
    const int u = (int)(p / d.Kb), ii = (int)(p % d.Kb);
    const bool live = ii < u_n[u - u_first];
    int blk = live ? sel[(size_t)u * d.Kb + ii] : -1;
    int slot = live ? slot_of_sel[(size_t)u * d.Kb + ii] : 0;
    if (live && (blk < 0 || blk >= n_blocks_of(u_len[u - u_first], d.bs) || slot < 0 || slot >= d.C)) {
      set_error(L.err, KVS_ERR_BAD_INDEX);
      blk = -1;
      slot = 0;
    }
    m_blk[i] = blk;
    m_slot[i] = slot;
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ------------------------------------------------------------------ producer
    if (lane != 0) return;
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
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
        } else {
          tma_load_2d(st, &tmK, 0, y, &full[s]);
          tma_load_2d(st + 16 * 128, &tmK, 64, y, &full[s]);
          tma_load_2d(st + kTile, &tmV, 0, y, &full[s]);
          tma_load_2d(st + kTile + 16 * 128, &tmV, 64, y, &full[s]);
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
  int k = 0;          // position in the CTA's tile sequence
  bool ok = true;
  for (int u = u_first; u <= u_last; ++u) {
    const int r = u / d.Hkv, h = u % d.Hkv;
    const int len = u_len[u - u_first];
    // queries of the group as m16n8k16 A fragments (rows >= G are zero)
    uint32_t qa[D / 16][4];
    {
      const int g0 = lane >> 2, g1 = g0 + 8, c2 = (lane & 3) * 2;
      const uint32_t* q0 = reinterpret_cast<const uint32_t*>(q + ((size_t)r * d.Hq + h * G + g0) * D);
      const uint32_t* q1 = reinterpret_cast<const uint32_t*>(q + ((size_t)r * d.Hq + h * G + g1) * D);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qa[ks][0] = g0 < G ? q0[(ks * 16 + c2) >> 1] : 0u;
        qa[ks][1] = (!ROWS8 && g1 < G) ? q1[(ks * 16 + c2) >> 1] : 0u;
        qa[ks][2] = g0 < G ? q0[(ks * 16 + 8 + c2) >> 1] : 0u;
        qa[ks][3] = (!ROWS8 && g1 < G) ? q1[(ks * 16 + 8 + c2) >> 1] : 0u;
      }
    }
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
    float oacc[D / 8][4];
#pragma unroll
    for (int x = 0; x < D / 8; ++x) oacc[x][0] = oacc[x][1] = oacc[x][2] = oacc[x][3] = 0.f;

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
          // widen the stage's K and V codes into this warp's bf16 staging (same swizzled layout as a
          // bf16 stage), then release the stage
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
            *reinterpret_cast<uint4*>(dst + sw128_offset(row, c16 * 16, 16)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(dst + sw128_offset(row, c16 * 16 + 8, 16)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
          kt = stg;
        }
        const unsigned char* vt = kt + kTile;
        const int valid_rows = rows - sub * 16;     // tokens of this tile before the context end
        // S = Q K^T
        float sacc[2][4];
#pragma unroll
        for (int nn = 0; nn < 2; ++nn) sacc[nn][0] = sacc[nn][1] = sacc[nn][2] = sacc[nn][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t b0, b1, b2, b3;
          const int trow = (lane & 7) + (lane >> 4) * 8;
          const int kcol = ks * 16 + ((lane >> 3) & 1) * 8;
          ldmatrix_x4(b0, b1, b2, b3, kt + sw128_offset(trow, kcol, 16));
          mma_bf16_16816(sacc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          mma_bf16_16816(sacc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
        // online softmax in the log2 domain; tokens past the context end are masked
        float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
        for (int nn = 0; nn < 2; ++nn)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int tok = nn * 8 + (lane & 3) * 2 + e;
            const bool valid = tok < valid_rows;
            const float slo = valid ? sacc[nn][e] * sl2 : -INFINITY;
            const float shi = valid ? sacc[nn][2 + e] * sl2 : -INFINITY;
            sacc[nn][e] = slo;
            sacc[nn][2 + e] = shi;
            mx_lo = fmaxf(mx_lo, slo);
            mx_hi = fmaxf(mx_hi, shi);
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
        for (int nn = 0; nn < 2; ++nn)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float plo = mn_lo == -INFINITY ? 0.f : exp2f(sacc[nn][e] - mn_lo);
            const float phi = mn_hi == -INFINITY ? 0.f : exp2f(sacc[nn][2 + e] - mn_hi);
            sacc[nn][e] = plo;
            sacc[nn][2 + e] = phi;
            ps_lo += plo;
            ps_hi += phi;
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
        for (int nd = 0; nd < D / 8; nd += 2) {
          oacc[nd][0] *= al_lo; oacc[nd][1] *= al_lo; oacc[nd][2] *= al_hi; oacc[nd][3] *= al_hi;
          oacc[nd + 1][0] *= al_lo; oacc[nd + 1][1] *= al_lo; oacc[nd + 1][2] *= al_hi; oacc[nd + 1][3] *= al_hi;
          uint32_t b0, b1, b2, b3;
          const int trow = (lane & 7) + ((lane >> 3) & 1) * 8;
          const int col = nd * 8 + (lane >> 4) * 8;
          ldmatrix_x4_trans(b0, b1, b2, b3, vt + sw128_offset(trow, col, 16));
          mma_bf16_16816(oacc[nd], ph[0], ph[1], ph[2], ph[3], b0, b1);
          mma_bf16_16816(oacc[nd], pl[0], pl[1], pl[2], pl[3], b0, b1);
          mma_bf16_16816(oacc[nd + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
          mma_bf16_16816(oacc[nd + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
        }
        __syncwarp();
        if (!FP8 && lane == 0) mbar_arrive(&empty[s]);
      }
    }
    // partial state of this warp for unit u
    const int c0 = (int)(((long long)u * d.Kb) / plan.per_cta);
    const int c1 = min(plan.n_cta - 1, (int)(((long long)(u + 1) * d.Kb - 1) / plan.per_cta));
    const size_t base = (size_t)u * plan.max_segs * kConsumers;
    const size_t pidx = base + (size_t)(c - c0) * kConsumers + warp;
    const int row_lo = lane >> 2, row_hi = row_lo + 8;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int row = hh ? row_hi : row_lo;
      if (row >= G) continue;
      float* dst = L.attn_part + (pidx * G + row) * D;
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        const int col = nd * 8 + (lane & 3) * 2;
        *reinterpret_cast<float2*>(dst + col) = make_float2(oacc[nd][hh * 2], oacc[nd][hh * 2 + 1]);
      }
      if ((lane & 3) == 0)
        *reinterpret_cast<float2*>(L.attn_ml + (pidx * G + row) * 2) = make_float2(hh ? m_hi : m_lo, hh ? l_hi : l_lo);
    }
    // Count this CTA's partials of unit u; the last CTA of the unit to finish merges them:
    // o = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p, partials in ascending order, one warp per
    // q head, 4 columns per lane.  The counter goes back to 0 for the next launch.
    __threadfence();
    named_bar_sync(1, kConsumers * 32);
    if (tid == 0) *last_flag = atomicAdd(&L.unit_done[u], 1u) == (unsigned)(c1 - c0);
    named_bar_sync(1, kConsumers * 32);
    if (*last_flag) {
      __threadfence();
      const int np = (c1 - c0 + 1) * kConsumers;
      const int r_out = u / d.Hkv, h_out = u % d.Hkv;
      for (int g = warp; g < G; g += kConsumers) {
        float M = -INFINITY;
        for (int p = lane; p < np; p += 32) M = fmaxf(M, __ldcg(L.attn_ml + ((base + p) * G + g) * 2));
#pragma unroll
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float lpart = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q0 = 0; q0 < np; q0 += 32) {
          float wgt = 0.f;
          if (q0 + lane < np) {
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(L.attn_ml + ((base + q0 + lane) * G + g) * 2));
            wgt = (M == -INFINITY || ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
            lpart += wgt * ml.y;
          }
          const int nj = min(32, np - q0);
          // eight partials' loads in flight at a time (they are independent; only the sums chain)
          for (int j0 = 0; j0 < nj; j0 += 8) {
            float4 x[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              x[k] = j0 + k < nj ? __ldcg(reinterpret_cast<const float4*>(L.attn_part + ((base + q0 + j0 + k) * G + g) * D) + lane)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float wj = __shfl_sync(0xffffffffu, wgt, (j0 + k) & 31);
              if (j0 + k < nj) {
                acc.x += wj * x[k].x;
                acc.y += wj * x[k].y;
                acc.z += wj * x[k].z;
                acc.w += wj * x[k].w;
              }
            }
          }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) lpart += __shfl_xor_sync(0xffffffffu, lpart, o);
        const float inv = lpart > 0.f ? (FP8 ? d.v_scale / lpart : 1.f / lpart) : 0.f;
        float4 res = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        reinterpret_cast<float4*>(out + ((size_t)r_out * d.Hq + h_out * G + g) * d.dv)[lane] = res;
      }
      if (tid == 0) L.unit_done[u] = 0u;
    }
  }
  if (!ok) set_error(L.err, KVS_ERR_TIMEOUT);
}

int sm_count() { return device_sm_count(); }

}  // namespace

int attention_tma_supported(const Dims& d) {
  return !d.v_shares_k && d.dk == D && d.dv == D && d.G <= 16 && d.bs % 16 == 0;
}

// Partial-result slots per unit the TMA path needs (segments x consumer warps).
int attention_tma_partials(const Dims& d) { return make_plan(d, sm_count()).max_segs * kConsumers; }

cudaError_t launch_attention_tma(const Dims& d, const Layer& L, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                 const __nv_bfloat16* q, const int* sel, const int* slot_of_sel, const int* nsel,
                                 const int* ctx_len, float* out, cudaStream_t s) {
  Plan plan = make_plan(d, sm_count());
  auto go = [&](auto kern, int smem) {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(plan.n_cta), dim3((kConsumers + 1) * 32), (size_t)smem, s, *tmK, *tmV, d, L, q, sel,
                      slot_of_sel, nsel, ctx_len, out, plan);
  };
  cudaError_t e;
  if (d.fp8)
    e = d.G <= 8 ? go(attn_tma_kernel<true, true>, Smem<true>::kTotal) : go(attn_tma_kernel<false, true>, Smem<true>::kTotal);
  else
    e = d.G <= 8 ? go(attn_tma_kernel<true, false>, Smem<false>::kTotal)
                 : go(attn_tma_kernel<false, false>, Smem<false>::kTotal);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvs
