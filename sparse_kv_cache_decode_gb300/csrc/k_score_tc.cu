// Block scoring on the 5th-generation tensor cores (tcgen05, sm_103a).
//
//   S^T (128 blocks x N rows) = IK (128 blocks x d_k) . Q^T (d_k x N rows),   s[b] = scale * max_row S
//
// Each CTA serves one unit: all its threads first write the unit's scoring rows into shared
// memory (K-major, 128-byte swizzle), then a contiguous range of the unit's 128-block tiles is
// processed by three roles:
//   warp 0   one lane streams the index tiles in 64-column chunks with 2D tensor loads into a
//            ring of stages (one mbarrier pair per stage);
//   warp 1   allocates the tensor memory, and one lane issues tcgen05.mma (M = 128, N = rows
//            padded to 16, K = 16 per instruction) into one of two fp32 accumulators in tensor
//            memory, releasing stages and accumulators with tcgen05.commit;
//   warps 2-5 read the accumulator rows (one TMEM lane per block) with tcgen05.ld, take the max
//            over the valid scoring rows and store the scaled score.
// Every wait is bounded by the context's timeout (KVS_ERR_TIMEOUT); the tensor memory is always
// released.
#include <cuda.h>

#include "kvs_common.cuh"
#include "kvs_ptx.cuh"

namespace kvs {

namespace {

constexpr int kTileM = 128;
constexpr int kChunk = 64;                         // d_k columns per stage (128 bytes)
constexpr int kChunkBytes = kTileM * kChunk * 2;  // 16 KiB
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kMaxSmem = 227 * 1024;
// No shared memory is kept free for a concurrent fetch CTA: with 128 scoring rows of 576 dims the
// staged rows leave room for 4 or 5 ring stages, and the fifth is worth more (per 16-layer MLA
// step, 3 / 4 / 5 stages: 7.89 / 7.21 / 7.13 ms of scoring, 0.72 / 0.79 / 0.80 of HBM).
constexpr int kSmemLeft = 0;

struct TcPlan {
  int n_rows, n_pad, kc, stages, q_bytes, tiles_per_unit, ctas_per_unit, per_cta, n_cta, tmem_cols, smem;
};

TcPlan make_tc_plan(const Dims& d, int nq, int n_sm) {
  TcPlan p;
  p.n_rows = nq * d.G;
  p.n_pad = ((p.n_rows + 15) / 16) * 16;
  p.kc = d.didx / kChunk;
  p.q_bytes = p.kc * p.n_pad * 128;
  const int fixed = 1024 + p.q_bytes + 512;
  p.stages = (kMaxSmem - kSmemLeft - fixed) / kChunkBytes;
  if (p.stages > 8) p.stages = 8;
  // each CTA serves one unit (its scoring rows are loaded once): the units' tiles are split over
  // floor(SMs / units) CTAs each, so every CTA fits in one wave
  p.tiles_per_unit = (d.nb_max + kTileM - 1) / kTileM;
  p.ctas_per_unit = n_sm / d.U;
  if (p.ctas_per_unit < 1) p.ctas_per_unit = 1;
  if (p.ctas_per_unit > p.tiles_per_unit) p.ctas_per_unit = p.tiles_per_unit;
  p.per_cta = (p.tiles_per_unit + p.ctas_per_unit - 1) / p.ctas_per_unit;
  p.ctas_per_unit = (p.tiles_per_unit + p.per_cta - 1) / p.per_cta;
  p.n_cta = d.U * p.ctas_per_unit;
  int cols = 32;
  while (cols < 2 * p.n_pad) cols <<= 1;
  p.tmem_cols = cols;
  p.smem = fixed + p.stages * kChunkBytes;
  return p;
}

__global__ void __launch_bounds__(kThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tm_idx, Dims d, const __nv_bfloat16* __restrict__ q, int nq,
                    const int* __restrict__ ctx_len, float* __restrict__ scores, TcPlan plan, unsigned* err) {
  kvs_pdl_entry();
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* a_st = smem;                                   // stages x 16 KiB
  unsigned char* qbuf = smem + plan.stages * kChunkBytes;       // kc x n_pad x 128 B
  uint64_t* full = reinterpret_cast<uint64_t*>(qbuf + plan.q_bytes);
  uint64_t* empty = full + 8;
  uint64_t* acc_full = empty + 8;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drained = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drained + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = blockIdx.x / plan.ctas_per_unit;
  const int t0 = (blockIdx.x - u * plan.ctas_per_unit) * plan.per_cta;
  const int len = ctx_len[u / d.Hkv];
  const int nb = (len < 0 || len > d.max_ctx) ? 0 : n_blocks_of(len, d.bs);
  const int t1 = min(min(plan.tiles_per_unit, t0 + plan.per_cta), (nb + kTileM - 1) / kTileM);
  const uint64_t timeout_ns = (uint64_t)d.timeout_us * 1000ull;
  const int S = plan.stages;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiWarps);
    }
    mbar_init(drained, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, plan.tmem_cols);
  // the unit's scoring rows (rows >= n_rows zero), 8 loads in flight per thread
  {
    const int r = u / d.Hkv, h = u % d.Hkv;
    const int ch = d.didx / 8;                         // 16-byte chunks per (staged) row
    const int total = plan.n_pad * ch;
    for (int base = tid; base < total; base += kThreads * 8) {
      uint4 v[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const int i = base + x * kThreads;
        v[x] = make_uint4(0, 0, 0, 0);
        const int row = i / ch;
        if (i < total && row < plan.n_rows) {
          const int j = row / d.G, g = row - j * d.G;
          v[x] = score_row_chunk(q + (((size_t)r * nq + j) * d.Hq + h * d.G + g) * d.dk, i - row * ch, d);
        }
      }
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const int i = base + x * kThreads;
        if (i < total) {
          const int row = i / ch, c16 = i - row * ch;
          const int kc = c16 >> 3, c = c16 & 7;
          *reinterpret_cast<uint4*>(qbuf + kc * plan.n_pad * 128 + row * 128 + ((c ^ (row & 7)) << 4)) = v[x];
        }
      }
    }
    fence_proxy_async_smem();                          // generic writes -> visible to the tensor cores
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() {
    set_error(err, KVS_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ loader
    int k = 0;
    if (lane == 0) {
      tma_prefetch_desc(&tm_idx);
      bool ok = true;
      for (int ti = t0; ti < t1 && ok; ++ti) {
        for (int kc = 0; kc < plan.kc; ++kc, ++k) {
          const int s = k % S;
          if (k >= S && !mbar_wait(&empty[s], ((k / S) & 1) ^ 1, timeout_ns)) { fail(); ok = false; break; }
          if (*abort_flag) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], kChunkBytes);
          tma_load_2d(a_st + s * kChunkBytes, &tm_idx, kc * kChunk, u * d.nb_max + ti * kTileM, &full[s]);
        }
      }
      // no tensor load may still be writing this CTA's shared memory when it exits (a fixed bound,
      // independent of the caller's timeout)
      for (int j = max(0, k - S); j < k; ++j) mbar_wait(&full[j % S], (j / S) & 1, kDrainTimeoutNs);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTileM, plan.n_pad);
      int k = 0, acc_n = 0;
      bool ok = true;
      for (int ti = t0; ti < t1 && ok; ++ti) {
        const int buf = acc_n & 1;
        if (acc_n >= 2 && !mbar_wait(&acc_empty[buf], ((acc_n >> 1) & 1) ^ 1, timeout_ns)) { fail(); break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(buf * plan.n_pad);
        for (int kc = 0; kc < plan.kc; ++kc, ++k) {
          const int s = k % S;
          if (!mbar_wait(&full[s], (k / S) & 1, timeout_ns)) { fail(); ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(a_st + s * kChunkBytes);
          const uint32_t b0 = smem_u32(qbuf + kc * plan.n_pad * 128);
#pragma unroll
          for (int k16 = 0; k16 < kChunk / 16; ++k16)
            tc_mma_f16(d_tmem, smem_desc_sw128(a0 + k16 * 32), smem_desc_sw128(b0 + k16 * 32), idesc,
                       (kc | k16) != 0);
          tc_commit(&empty[s]);
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
        ++acc_n;
      }
      // every product issued by this thread has finished before the tensor memory is released
      tc_commit(drained);
      mbar_wait(drained, 0, kDrainTimeoutNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    const int lane_base = (warp & 3) * 32;
    const int row = lane_base + lane;
    int acc_n = 0;
    for (int ti = t0; ti < t1; ++ti) {
      const int buf = acc_n & 1;
      bool got = true;
      if (lane == 0) got = mbar_wait(&acc_full[buf], (acc_n >> 1) & 1, timeout_ns);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)lane_base << 16) + (uint32_t)(buf * plan.n_pad);
      float m = -INFINITY;
      for (int c0 = 0; c0 < plan.n_pad; c0 += 16) {
        float v[16];
        tmem_ld16(taddr + c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (c0 + i < plan.n_rows) m = fmaxf(m, v[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
      const int b = ti * kTileM + row;
      if (b < nb) scores[(size_t)u * d.nb_max + b] = __fmul_rn(d.scale, m);
      ++acc_n;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, plan.tmem_cols);
  }
}

int sm_count_tc() { return device_sm_count(); }

}  // namespace

int score_tc_supported(const Dims& d, int nq) {
  // the tensor-memory path pays off for wide contractions (many scoring rows per index row)
  if (d.didx % kChunk != 0 || nq * d.G > 256 || nq * d.G < 64) return 0;
  TcPlan p = make_tc_plan(d, nq, sm_count_tc());
  return p.stages >= 2;
}

cudaError_t launch_score_tc(const Dims& d, const __nv_bfloat16* index, const __nv_bfloat16* q, int nq,
                            const int* ctx_len, float* scores, unsigned* err, cudaStream_t s) {
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(score_tc_kernel), kMaxSmem);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tm;
  if (!make_tmap_2d(&tm, const_cast<__nv_bfloat16*>(index), (uint64_t)d.didx, (uint64_t)d.U * d.nb_max, kChunk, kTileM))
    return cudaErrorInvalidValue;
  TcPlan plan = make_tc_plan(d, nq, sm_count_tc());
  launch_pdl(score_tc_kernel, dim3(plan.n_cta), dim3(kThreads), plan.smem, s, tm, d, q, nq, ctx_len, scores, plan, err);
  return cudaGetLastError();
}

}  // namespace kvs
