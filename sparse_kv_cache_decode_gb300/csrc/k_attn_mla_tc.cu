// MLA decode attention on the 5th-generation tensor cores (tcgen05, sm_103a): 128 query heads
// share one latent KV row per token (d_k = 576: 512 latent + 64 rope dims; V = the first 512 dims
// of the same row), as in the token-level sparse selection of DeepSeek-style MLA models.
//
// One CTA serves (split of the unit's selection, unit, value half z).  Per tile of 32 tokens:
//   S (128 heads x 32 tokens, fp32, tensor memory)  = Q (128 x 576) . K_tile^T
//   P = 2^(S * scale * log2 e - m) split into bf16 hi + lo parts, written back to tensor memory
//   O (128 heads x 256 dims, fp32, tensor memory)  += P_hi . V_tile[:, z half] + P_lo . V_tile[:, z half]
// The 512 value dims do not fit tensor memory beside S, so the two halves of O are two CTAs, each
// computing S the same way (same inputs, same instruction sequence, so bit-identical).
//
// Products of one accumulator run one after another, and a 128 x 32 x 16 product is short, so one
// chain of 36 products (576 dims) would leave the tensor pipe idle between them: S is summed in 4
// independent chains (chain c takes the 16-dim steps 4i + c) that the softmax adds.  Q's first 128
// dims are an A operand in tensor memory, the other 448 in shared memory beside a 3-stage ring of
// token tiles.  Roles (256 threads):
//   warps 0-2  warp w gathers tiles w, w + 3, ... into stage w (the tile's token rows are slot
//              pool rows, scattered) with 16-byte cp.async as K-major 128-byte-swizzled chunks of
//              64 dims, so up to three tiles are in flight;
//   warp 3     allocates tensor memory; one lane issues QK of tile j+1 before PV of tile j, so
//              the softmax of one tile overlaps the products of the next;
//   warps 4-7  load Q (while the first tiles arrive), then one thread per head: read its S row,
//              update its running max with lazy rescaling (O is rescaled in tensor memory only when
//              a tile's max exceeds the reference max by more than 2^8, so every P stays <= 256),
//              write P, and finally write O.
// The value tile is read by the PV product as an MN-major operand of the same swizzled storage.
// With several splits, the last CTA of a (unit, half) to finish merges the splits' partial states
// (a per-unit completion counter).  Every wait is bounded by the context's timeout
// (KVS_ERR_TIMEOUT); tensor memory is always freed.
#include <algorithm>

#include "kvs_common.cuh"
#include "kvs_ptx.cuh"

namespace kvs {

namespace {
namespace mtc {
constexpr int DK = 576, DV = 512, H = 128;
constexpr int NTOK = 32;                            // tokens per tile
constexpr int KC = DK / 64;                         // 64-dim chunks of a row (128 bytes each)
constexpr int KC_TM = 2;                            // chunks of Q held in tensor memory (dims 0-127)
constexpr int NCHAIN = 4;                           // independent accumulator chains of S
constexpr int DVZ = DV / 2;                         // value dims per CTA
constexpr int CHUNK = NTOK * 128;                   // one 64-dim chunk of a tile (4 KiB)
constexpr int TILE = KC * CHUNK;                    // 36 KiB
constexpr int QCHUNK = H * 128;                     // one 64-dim chunk of Q (16 KiB)
constexpr int QS_BYTES = (KC - KC_TM) * QCHUNK;     // Q dims 128-575 in shared memory (112 KiB)
constexpr int STAGES = 3;                           // one per producer warp
constexpr int MMA_WARP = STAGES;
constexpr int SOFT0 = STAGES + 1;                   // first softmax warp (its warp index % 4 = TMEM lane quarter)
constexpr int MAX_TOK = 512;                        // tokens per CTA (their pool rows staged in shared memory)
constexpr int SOFT = 128;
constexpr int THREADS = SOFT0 * 32 + SOFT;
constexpr int NWARPS = THREADS / 32;
constexpr int OFF_TILES = QS_BYTES;
constexpr int OFF_ROWS = OFF_TILES + STAGES * TILE;
constexpr int OFF_BAR = OFF_ROWS + MAX_TOK * 4;
constexpr int SMEM = OFF_BAR + 256 + 1024;          // + slack for 1024-byte alignment
// tensor memory columns: O, S (4 chains), P (2 buffers of hi 16 + lo 16), Q dims 0-127 (bf16 pairs)
constexpr uint32_t T_O = 0, T_S = 256, T_P = 384, T_Q = 448, TMEM_COLS = 512;
static_assert(T_S + NCHAIN * NTOK == T_P && T_P + 64 == T_Q && T_Q + KC_TM * 32 == TMEM_COLS, "tensor memory plan");
static_assert(SMEM <= 227 * 1024, "shared memory plan");
static_assert(SOFT0 % 4 == 0, "softmax warps must cover the four TMEM lane quarters in order");
constexpr float kMaxGrowth = 8.f;                   // log2 of the largest P before O is rescaled
constexpr float kLog2e = 1.4426950408889634f;
}  // namespace mtc

__global__ void __launch_bounds__(mtc::THREADS, 1)
    attn_mla_tc_kernel(Dims d, Layer L, const __nv_bfloat16* __restrict__ q, const int* __restrict__ sel,
                       const int* __restrict__ slot_of_sel, const int* __restrict__ nsel,
                       const int* __restrict__ ctx_len, float* __restrict__ out, int n_split, int blocks_per_split) {
  using namespace mtc;
  kvs_pdl_entry();
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* qs = smem;
  unsigned char* tiles = smem + OFF_TILES;
  int* rows = reinterpret_cast<int*>(smem + OFF_ROWS);          // pool row of each token, -1 masked
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* full = bars;           // [3] producer warp (32 arrivals)
  uint64_t* empty = bars + 3;      // [3] tcgen05.commit after the tile's PV
  uint64_t* s_full = bars + 6;     // commit after QK
  uint64_t* s_free = bars + 7;     // softmax warps (4 arrivals) have read S
  uint64_t* p_full = bars + 8;     // [2] softmax warps have written P (and rescaled O)
  uint64_t* pv_done = bars + 10;   // [2] commit after PV
  uint64_t* drained = bars + 12;
  uint64_t* q_ready = bars + 13;   // softmax warps (4 arrivals) have placed Q
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* last_flag = const_cast<int*>(abort_flag + 1);

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
  const int ntok = (i1 - i0) * d.bs;
  const int T = (ntok + NTOK - 1) / NTOK;
  const uint64_t timeout_ns = (uint64_t)d.timeout_us * 1000ull;
  const __nv_bfloat16* qrow0 = q + ((size_t)r * d.Hq + (size_t)h * d.G) * DK;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 32);
      mbar_init(&empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, SOFT / 32);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&p_full[b], SOFT / 32);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(drained, 1);
    mbar_init(q_ready, SOFT / 32);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == MMA_WARP) tmem_alloc(tmem_slot, TMEM_COLS);
  for (int t = tid; t < ntok; t += THREADS) {
    const int bi = t / d.bs, rr = t - bi * d.bs;
    const int slot = slot_of_sel[(size_t)u * d.Kb + i0 + bi];
    const int blk = sel[(size_t)u * d.Kb + i0 + bi];
    int row = -1;
    if (blk < 0 || blk >= n_blocks_of(len, d.bs) || slot < 0 || slot >= d.C) {   // reported, then masked
      if (rr == 0) set_error(L.err, KVS_ERR_BAD_INDEX);
    } else if (blk * d.bs + rr < len) {
      row = slot * d.bs + rr;
    }
    rows[t] = row;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() {
    set_error(L.err, KVS_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp < STAGES) {
    // ------------------------------------------------------------------ producers: warp w, stage w
    const __nv_bfloat16* kbase = L.kpool + (size_t)u * d.C * d.bs * DK;
    const int rq = lane >> 2, part = lane & 3;
    unsigned char* stage = tiles + warp * TILE;
    for (int j = warp; j < T; j += STAGES) {
      if (j >= STAGES) {
        if (!mbar_wait(&empty[warp], ((j / STAGES) & 1) ^ 1, timeout_ns)) { fail(); break; }
        if (*abort_flag) break;
      }
#pragma unroll 1
      for (int g8 = 0; g8 < NTOK / 8; ++g8) {
        const int trow = g8 * 8 + rq, t = j * NTOK + trow;
        const int prow = t < ntok ? rows[t] : -1;
        const __nv_bfloat16* src = kbase + (size_t)(prow < 0 ? 0 : prow) * DK;
        unsigned char* dst = stage + trow * 128;
#pragma unroll
        for (int i = 0; i < DK / 8 / 4; ++i) {
          const int c = part + 4 * i;
          cp_async16(dst + (c >> 3) * CHUNK + (((c & 7) ^ (trow & 7)) << 4), src + c * 8, prow < 0 ? 0 : 16);
        }
      }
      cp_async_commit();
      cp_async_wait_all();
      fence_proxy_async_smem();               // this lane's copies -> visible to the tensor cores
      mbar_arrive(&full[warp]);
    }
    cp_async_wait_all();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(H, NTOK);
      const uint32_t idesc_pv = idesc_bf16_f32(H, DVZ) | (1u << 16);   // B (the value tile) MN-major
      // descriptors advance with the start address (its field holds address / 16)
      const uint64_t dq0 = smem_desc_sw128(smem_u32(qs));
      bool ok = mbar_wait(q_ready, 0, timeout_ns);
      if (!ok) fail();
      for (int j = 0; j <= T && ok; ++j) {
        if (j < T) {
          const int s = j % STAGES;
          if (!mbar_wait(&full[s], (j / STAGES) & 1, timeout_ns)) { fail(); break; }
          if (j >= 1 && !mbar_wait(s_free, (j - 1) & 1, timeout_ns)) { fail(); break; }
          tc_fence_after();
          const uint64_t dk0 = smem_desc_sw128(smem_u32(tiles + s * TILE));
#pragma unroll
          for (int kc = 0; kc < KC; ++kc) {
#pragma unroll
            for (int c = 0; c < NCHAIN; ++c) {
              const uint64_t bdesc = dk0 + (uint64_t)((kc * CHUNK + c * 32) >> 4);
              const uint32_t acc = tmem + T_S + c * NTOK;
              if (kc < KC_TM)
                tc_mma_f16_ts(acc, tmem + T_Q + kc * 32 + c * 8, bdesc, idesc_qk, kc != 0);
              else
                tc_mma_f16(acc, dq0 + (uint64_t)(((kc - KC_TM) * QCHUNK + c * 32) >> 4), bdesc, idesc_qk, kc != 0);
            }
          }
          tc_commit(s_full);
        }
        if (j >= 1) {
          const int jj = j - 1, b = jj & 1, s = jj % STAGES;
          if (!mbar_wait(&p_full[b], (jj >> 1) & 1, timeout_ns)) { fail(); break; }
          tc_fence_after();
          // value dims [256 z, 256 z + 256) = chunks 4z .. 4z + 3 of the tile (64-dim blocks CHUNK
          // bytes apart), 16 tokens per product (two 8-row groups, 1024 bytes apart)
          const uint32_t tv = smem_u32(tiles + s * TILE + 4 * z * CHUNK);
#pragma unroll
          for (int kk = 0; kk < NTOK / 16; ++kk) {
            const uint64_t bdesc = smem_desc_sw128_mn(tv + kk * 2048, CHUNK, 1024);
            tc_mma_f16_ts(tmem + T_O, tmem + T_P + b * 32 + kk * 8, bdesc, idesc_pv, (jj | kk) != 0);
            tc_mma_f16_ts(tmem + T_O, tmem + T_P + b * 32 + 16 + kk * 8, bdesc, idesc_pv, 1);
          }
          tc_commit(&pv_done[b]);
          tc_commit(&empty[s]);
        }
        if (*abort_flag) ok = false;
      }
      // every product issued by this thread has finished before the tensor memory is released
      tc_commit(drained);
      mbar_wait(drained, 0, kDrainTimeoutNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ Q, then softmax + output
    const int lane_base = (warp & 3) * 32;
    const int head = lane_base + lane;                     // TMEM lane = head within the unit
    const uint32_t trow = tmem + ((uint32_t)lane_base << 16);
    {
      const int st = tid - SOFT0 * 32;
      // dims 128-575: K-major 128-byte-swizzled chunks of 64 dims in shared memory
      constexpr int QS_C16 = (KC - KC_TM) * 8;            // 16-byte chunks per row
      for (int i = st; i < H * QS_C16; i += SOFT) {
        const int row = i / QS_C16, c = i - row * QS_C16;
        cp_async16(qs + (c >> 3) * QCHUNK + row * 128 + (((c & 7) ^ (row & 7)) << 4),
                   qrow0 + (size_t)row * DK + KC_TM * 64 + c * 8, 16);
      }
      cp_async_commit();
      // dims 0-127 of this thread's head -> its tensor-memory lane (bf16 pairs, lower dim low)
      const uint4* src = reinterpret_cast<const uint4*>(qrow0 + (size_t)head * DK);
      uint4 x[KC_TM * 8];
#pragma unroll
      for (int i = 0; i < KC_TM * 8; ++i) x[i] = src[i];
#pragma unroll
      for (int cb = 0; cb < KC_TM; ++cb) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[4 * i] = __uint_as_float(x[cb * 8 + i].x);
          v[4 * i + 1] = __uint_as_float(x[cb * 8 + i].y);
          v[4 * i + 2] = __uint_as_float(x[cb * 8 + i].z);
          v[4 * i + 3] = __uint_as_float(x[cb * 8 + i].w);
        }
        tmem_st32(trow + T_Q + cb * 32, v);
      }
      tmem_wait_st();
      cp_async_wait_all();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_ready);
    }
    const float sl2 = d.scale * kLog2e;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    auto wait_all_lanes = [&](uint64_t* bar, unsigned parity) {
      bool got = true;
      if (lane == 0) got = mbar_wait(bar, parity, timeout_ns);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got && lane == 0) fail();
      return got;
    };
    for (int j = 0; j < T && ok; ++j) {
      const int b = j & 1;
      if (!wait_all_lanes(s_full, j & 1)) { ok = false; break; }
      tc_fence_after();
      float sv[32];
      tmem_ld32(trow + T_S, sv);
#pragma unroll
      for (int c = 1; c < NCHAIN; ++c) {
        float sc[32];
        tmem_ld32(trow + T_S + c * NTOK, sc);
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[i] += sc[i];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      float tmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < NTOK; ++i) {
        const int t = j * NTOK + i;
        const bool valid = t < ntok && rows[t] >= 0;
        sv[i] = valid ? sv[i] * sl2 : -INFINITY;
        tmax = fmaxf(tmax, sv[i]);
      }
      const bool grow = tmax > m + kMaxGrowth || (m == -INFINITY && tmax != -INFINITY);
      const float m_new = grow ? tmax : m;
      const float alpha = grow ? (m == -INFINITY ? 0.f : exp2f(m - m_new)) : 1.f;
      // O holds earlier tiles' products: rescale it (after the previous PV) where the reference grew
      if (__any_sync(0xffffffffu, grow && l > 0.f)) {
        if (!wait_all_lanes(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const float f = (grow && l > 0.f) ? alpha : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < DVZ; c0 += 32) {
          float ov[32];
          tmem_ld32(trow + T_O + c0, ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] *= f;
          tmem_st32(trow + T_O + c0, ov);
        }
        tmem_wait_st();
      }
      l *= alpha;
      m = m_new;
      // the P buffer of this tile was last read by the PV of tile j - 2
      if (j >= 2 && !wait_all_lanes(&pv_done[b], ((j - 2) >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      uint32_t ph[16], pl[16];
      float ps = 0.f;
#pragma unroll
      for (int i = 0; i < NTOK; i += 2) {
        const float p0 = m == -INFINITY ? 0.f : exp2f(sv[i] - m);
        const float p1 = m == -INFINITY ? 0.f : exp2f(sv[i + 1] - m);
        ps += p0 + p1;
        ph[i / 2] = pack_bf16x2(p0, p1);
        pl[i / 2] = pack_bf16x2(p0 - bf16_lo(ph[i / 2]), p1 - bf16_hi(ph[i / 2]));
      }
      l += ps;
      tmem_st16(trow + T_P + b * 32, ph);
      tmem_st16(trow + T_P + b * 32 + 16, pl);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[b]);
    }
    // the last PV, then O out: normalised (one split) or the split's partial state
    if (ok && T > 0 && !wait_all_lanes(&pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1)) ok = false;
    if (ok) {
      tc_fence_after();
      const int g = head;                                    // q head within the unit's group
      float* dst;
      float sc = 1.f;
      if (n_split == 1) {
        dst = out + ((size_t)r * d.Hq + (size_t)h * d.G + g) * d.dv + z * DVZ;
        sc = l > 0.f ? 1.f / l : 0.f;
      } else {
        dst = L.attn_part + (((size_t)u * n_split + split) * d.G + g) * d.dv + z * DVZ;
        // both halves write the same (bit-identical) state, so each half's merge reads its own
        *reinterpret_cast<float2*>(L.attn_ml + (((size_t)u * n_split + split) * d.G + g) * 2) = make_float2(m, l);
      }
#pragma unroll 1
      for (int c0 = 0; c0 < DVZ; c0 += 32) {
        float ov[32];
        if (T > 0) {
          tmem_ld32(trow + T_O + c0, ov);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(dst + c0 + i) = make_float4(ov[i] * sc, ov[i + 1] * sc, ov[i + 2] * sc, ov[i + 3] * sc);
      }
    }
    __threadfence();                        // the partial state is visible before the CTA is counted
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
  if (n_split == 1) return;
  // ---------------------------------------------------------------- merge of the splits (last CTA)
  // counter: low 16 bits count the finished CTAs of half 0, high 16 bits those of half 1
  if (tid == 0) {
    __threadfence();
    const unsigned one = z == 0 ? 1u : 65536u;
    const unsigned prev = atomicAdd(&L.unit_done[u], one);
    const unsigned mine = z == 0 ? (prev & 0xffffu) : (prev >> 16);
    *last_flag = mine == (unsigned)(n_split - 1);
    if (*last_flag) {
      atomicSub(&L.unit_done[u], one * (unsigned)n_split);   // 0 again for the next launch
      __threadfence();
    }
  }
  __syncthreads();
  if (!*last_flag) return;
  // the splits' (max, sum) -> per-split weights 2^(m_s - M) / sum_s 2^(m_s - M) l_s in shared
  // memory (the tile ring is free now), then every output float4 of the half as a weighted sum of
  // the splits' partial rows, sixteen loads in flight per thread
  float2* mls = reinterpret_cast<float2*>(tiles);                     // [n_split][128]
  float* wts = reinterpret_cast<float*>(tiles + (size_t)kAttnSplitMax * H * sizeof(float2));
  const float2* pml = reinterpret_cast<const float2*>(L.attn_ml) + (size_t)u * n_split * d.G;
  for (int i = tid; i < n_split * H; i += THREADS) mls[i] = __ldcg(pml + i);
  __syncthreads();
  if (tid < H) {
    float M = -INFINITY;
    for (int s = 0; s < n_split; ++s) M = fmaxf(M, mls[s * H + tid].x);
    float lsum = 0.f;
    for (int s = 0; s < n_split; ++s) {
      const float2 v = mls[s * H + tid];
      if (v.x != -INFINITY) lsum += exp2f(v.x - M) * v.y;
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    for (int s = 0; s < n_split; ++s) {
      const float ms = mls[s * H + tid].x;
      wts[s * H + tid] = ms == -INFINITY ? 0.f : exp2f(ms - M) * inv;
    }
  }
  __syncthreads();
  constexpr int F4 = DVZ / 4;                                         // float4 per head row half
  constexpr int ITEMS = H * F4;
  const float4* part = reinterpret_cast<const float4*>(L.attn_part + (size_t)u * n_split * d.G * d.dv + z * DVZ);
  float4* outv = reinterpret_cast<float4*>(out + ((size_t)r * d.Hq + (size_t)h * d.G) * d.dv + z * DVZ);
  const size_t split_f4 = (size_t)d.G * d.dv / 4, row_f4 = d.dv / 4;
  for (int base = tid; base < ITEMS; base += 4 * THREADS) {
    int gi[4], ci[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = min(base + k * THREADS, ITEMS - 1);
      gi[k] = i / F4;
      ci[k] = i - gi[k] * F4;
    }
    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < n_split; s0 += 4) {
      float4 x[4][4];
#pragma unroll
      for (int ss = 0; ss < 4; ++ss) {
        const int s = min(s0 + ss, n_split - 1);
#pragma unroll
        for (int k = 0; k < 4; ++k) x[ss][k] = __ldcg(part + s * split_f4 + gi[k] * row_f4 + ci[k]);
      }
#pragma unroll
      for (int ss = 0; ss < 4; ++ss) {
        if (s0 + ss < n_split) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float w = wts[(s0 + ss) * H + gi[k]];
            acc[k].x += w * x[ss][k].x;
            acc[k].y += w * x[ss][k].y;
            acc[k].z += w * x[ss][k].z;
            acc[k].w += w * x[ss][k].w;
          }
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (base + k * THREADS < ITEMS) outv[gi[k] * row_f4 + ci[k]] = acc[k];
  }
}

}  // namespace

int attention_mla_tc_split(const Dims& d, int* n_split_out, int* bps_out) {
  if (!(d.v_shares_k && d.dk == mtc::DK && d.dv == mtc::DV && d.G == mtc::H && !d.fp8)) return 0;
  if (d.bs > mtc::MAX_TOK) return 0;
  const int cap = mtc::MAX_TOK / d.bs;                          // blocks per CTA
  const int n_min = (d.Kb + cap - 1) / cap;
  // one CTA per SM (shared memory): fill one wave with (split, unit, half) CTAs, at least two
  // tiles of tokens per CTA
  const int fill = device_sm_count() / (2 * d.U);
  const int tiles = (d.Kb * d.bs + mtc::NTOK - 1) / mtc::NTOK;
  int n = std::max(n_min, std::min(fill, tiles / 2));
  n = std::max(n, 1);
  int bps = (d.Kb + n - 1) / n;
  n = (d.Kb + bps - 1) / bps;
  if (n > kAttnSplitMax) return 0;
  *n_split_out = n;
  *bps_out = bps;
  return 1;
}

int attention_mla_tc_supported(const Dims& d) {
  int n, bps;
  return attention_mla_tc_split(d, &n, &bps);
}

cudaError_t launch_attention_mla_tc(const Dims& d, const Layer& L, const __nv_bfloat16* q, const int* sel,
                                    const int* slot_of_sel, const int* nsel, const int* ctx_len, float* out,
                                    cudaStream_t s) {
  int n_split, bps;
  if (!attention_mla_tc_split(d, &n_split, &bps)) return cudaErrorInvalidValue;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(attn_mla_tc_kernel), mtc::SMEM);
  if (e != cudaSuccess) return e;
  launch_pdl(attn_mla_tc_kernel, dim3(n_split, d.U, 2), dim3(mtc::THREADS), mtc::SMEM, s, d, L, q, sel, slot_of_sel,
             nsel, ctx_len, out, n_split, bps);
  return cudaGetLastError();
}

}  // namespace kvs
