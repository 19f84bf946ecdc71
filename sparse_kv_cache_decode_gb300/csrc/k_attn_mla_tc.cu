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
// S is double-buffered in tensor memory, so the products of tile j+1 run while the softmax reads
// tile j, and summed in 2 accumulator chains (even and odd 16-dim steps) that the softmax adds.
// Q's first 128 dims are an A operand in tensor memory, the other 448 in shared memory beside a
// 3-stage ring of token tiles.  Roles (256 threads):
//   warps 0-2  warp w gathers tiles w, w + 3, ... into stage w (the tile's token rows are slot
//              pool rows, scattered) with 16-byte cp.async as K-major 128-byte-swizzled chunks of
//              64 dims, so up to three tiles are in flight;
//   warp 3     allocates tensor memory; one lane issues QK of tile j+1 before PV of tile j, so
//              the softmax of one tile overlaps the products of the next;
//   warps 4-7  load Q (while the first tiles arrive), then one thread per head: read its S row,
//              update its running max with lazy rescaling (O is rescaled in tensor memory only when
//              a tile's max exceeds the reference max by more than 2^8, so every P stays <= 256),
//              write P, and finally write O (one split) or send it to the cluster merge.
// The value tile is read by the PV product as an MN-major operand of the same swizzled storage.
// With several splits, the splits of a (unit, half) form a thread-block cluster: each CTA sends
// its O rows and (max, sum) straight from tensor memory to the CTA that owns those heads (its
// shared memory, through the cluster's distributed shared memory), and each CTA merges its share
// of the heads and writes them out.  Every wait is bounded by the context's timeout
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
constexpr int NCHAIN = 2;                           // accumulator chains of S (even / odd 16-dim steps)
constexpr int DVZ = DV / 2;                         // value dims per CTA
constexpr int CHUNK = NTOK * 128;                   // one 64-dim chunk of a tile (4 KiB)
constexpr int TILE = KC * CHUNK;                    // 36 KiB
constexpr int QCHUNK = H * 128;                     // one 64-dim chunk of Q (16 KiB)
constexpr int QS_BYTES = (KC - KC_TM) * QCHUNK;     // Q dims 128-575 in shared memory (112 KiB)
constexpr int STAGES = 3;                           // one per producer warp
constexpr int MMA_WARP = STAGES;
constexpr int SOFT0 = STAGES + 1;                   // first softmax warp (its warp index % 4 = TMEM lane quarter)
constexpr int MAX_TOK = 512;                        // tokens per CTA (their pool rows staged in shared memory)
constexpr int MAX_SPLIT = 8;                        // CTAs per cluster (portable limit)
constexpr int SOFT = 128;
constexpr int THREADS = SOFT0 * 32 + SOFT;
constexpr int OFF_TILES = QS_BYTES;
constexpr int OFF_ROWS = OFF_TILES + STAGES * TILE;
constexpr int OFF_BAR = OFF_ROWS + MAX_TOK * 4;
constexpr int SMEM = OFF_BAR + 256 + 1024;          // + slack for 1024-byte alignment
// tensor memory columns: O, S (2 buffers x 2 chains), P (2 buffers of hi 16 + lo 16), Q dims 0-127
// (bf16 pairs)
constexpr uint32_t T_O = 0, T_S = 256, T_P = 384, T_Q = 448, TMEM_COLS = 512;
constexpr uint32_t S_BUF = NCHAIN * NTOK;           // columns of one S buffer
static_assert(T_S + 2 * S_BUF == T_P && T_P + 64 == T_Q && T_Q + KC_TM * 32 == TMEM_COLS, "tensor memory plan");
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
  uint64_t* s_full = bars + 6;     // [2] commit after QK
  uint64_t* s_free = bars + 8;     // [2] softmax warps (4 arrivals) have read S
  uint64_t* p_full = bars + 10;    // [2] softmax warps have written P (and rescaled O)
  uint64_t* pv_done = bars + 12;   // [2] commit after PV
  uint64_t* drained = bars + 14;
  uint64_t* q_ready = bars + 15;   // softmax warps (4 arrivals) have placed Q
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

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
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], SOFT / 32);
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
  float sm_m = -INFINITY, sm_l = 0.f;        // this thread's head state, handed to the merge
  bool sm_ok = false;

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
          const int sb = j & 1;
          if (j >= 2 && !mbar_wait(&s_free[sb], ((j >> 1) - 1) & 1, timeout_ns)) { fail(); break; }
          tc_fence_after();
          const uint64_t dk0 = smem_desc_sw128(smem_u32(tiles + s * TILE));
          const uint32_t sacc = tmem + T_S + sb * S_BUF;
#pragma unroll
          for (int kc = 0; kc < KC; ++kc) {
#pragma unroll
            for (int k16 = 0; k16 < 4; ++k16) {
              const uint64_t bdesc = dk0 + (uint64_t)((kc * CHUNK + k16 * 32) >> 4);
              const uint32_t acc = sacc + (k16 & 1) * NTOK;
              const uint32_t first = kc == 0 && k16 < NCHAIN;
              if (kc < KC_TM)
                tc_mma_f16_ts(acc, tmem + T_Q + kc * 32 + k16 * 8, bdesc, idesc_qk, !first);
              else
                tc_mma_f16(acc, dq0 + (uint64_t)(((kc - KC_TM) * QCHUNK + k16 * 32) >> 4), bdesc, idesc_qk, !first);
            }
          }
          tc_commit(&s_full[sb]);
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
      // token i of the tile is valid when bit i is set (lane i looks its token up)
      const int tl = j * NTOK + lane;
      const unsigned vmask = __ballot_sync(0xffffffffu, tl < ntok && rows[tl] >= 0);
      if (!wait_all_lanes(&s_full[b], (j >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      float sv[32];
      {
        float s2[2 * NTOK];
        tmem_ld64(trow + T_S + b * S_BUF, s2);
#pragma unroll
        for (int i = 0; i < NTOK; ++i) sv[i] = s2[i] + s2[NTOK + i];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[b]);
      float tmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < NTOK; ++i) {
        sv[i] = (vmask >> i) & 1u ? sv[i] * sl2 : -INFINITY;
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
    // the last PV
    if (ok && T > 0 && !wait_all_lanes(&pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1)) ok = false;
    tc_fence_after();
    if (n_split == 1 && ok) {
      const float sc = l > 0.f ? 1.f / l : 0.f;
      float* dst = out + ((size_t)r * d.Hq + (size_t)h * d.G + head) * d.dv + z * DVZ;
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
    if (!ok) {                                // reported; the partial state sent below is empty
      m = -INFINITY;
      l = 0.f;
    }
    sm_m = m;
    sm_l = l;
    sm_ok = ok && T > 0;
  }
  if (n_split > 1) {
    // ---------------------------------------------------------------- merge over the cluster
    // head g belongs to cluster rank g * n / 128; each rank's heads arrive in its shared memory
    // (the Q and ring area, free once every CTA of the cluster has left its main loop) as
    // [source rank][head - first head][256] floats and [source rank][head - first head] (max, sum)
    const uint32_t me = cluster_ctarank();
    const int rows_max = (H + n_split - 1) / n_split;
    float* oslots = reinterpret_cast<float*>(smem);
    float2* mlslots = reinterpret_cast<float2*>(smem + (size_t)n_split * rows_max * DVZ * 4);
    float* wts = reinterpret_cast<float*>(mlslots + n_split * rows_max);
    __syncwarp();
    cluster_sync();
    if (warp >= SOFT0) {
      const int head = (warp & 3) * 32 + lane;
      const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      const int owner = head * n_split / H;
      const int first = (owner * H + n_split - 1) / n_split;
      const int row = (int)me * rows_max + (head - first);
      const uint32_t ro = mapa_shared(smem_u32(oslots + (size_t)row * DVZ), (uint32_t)owner);
#pragma unroll 1
      for (int c0 = 0; c0 < DVZ; c0 += 32) {
        float ov[32];
        if (sm_ok) {
          tmem_ld32(trow + T_O + c0, ov);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 32; i += 4) st_cluster_f4(ro + (c0 + i) * 4, ov[i], ov[i + 1], ov[i + 2], ov[i + 3]);
      }
      st_cluster_f2(mapa_shared(smem_u32(mlslots + row), (uint32_t)owner), sm_m, sm_l);
    }
    cluster_sync();
    const int first = ((int)me * H + n_split - 1) / n_split;
    const int cnt = (((int)me + 1) * H + n_split - 1) / n_split - first;
    // weights 2^(m_k - M) / sum_k 2^(m_k - M) l_k of each source rank k, per head of this rank
    if (tid < cnt) {
      float M = -INFINITY;
      for (int k = 0; k < n_split; ++k) M = fmaxf(M, mlslots[k * rows_max + tid].x);
      float lsum = 0.f;
      for (int k = 0; k < n_split; ++k) {
        const float2 v = mlslots[k * rows_max + tid];
        if (v.x != -INFINITY) lsum += exp2f(v.x - M) * v.y;
      }
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      for (int k = 0; k < n_split; ++k) {
        const float mk = mlslots[k * rows_max + tid].x;
        wts[k * rows_max + tid] = mk == -INFINITY ? 0.f : exp2f(mk - M) * inv;
      }
    }
    __syncthreads();
    constexpr int F4 = DVZ / 4;
    const float4* os4 = reinterpret_cast<const float4*>(oslots);
    float4* outv = reinterpret_cast<float4*>(out + ((size_t)r * d.Hq + (size_t)h * d.G + first) * d.dv + z * DVZ);
    for (int i = tid; i < cnt * F4; i += THREADS) {
      const int g = i / F4, c4 = i - g * F4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k = 0; k < n_split; ++k) {
        const float w = wts[k * rows_max + g];
        const float4 x = os4[(size_t)(k * rows_max + g) * F4 + c4];
        acc.x += w * x.x;
        acc.y += w * x.y;
        acc.z += w * x.z;
        acc.w += w * x.w;
      }
      outv[(size_t)g * (d.dv / 4) + c4] = acc;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
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
  int n = std::max(n_min, std::min(std::min(fill, tiles / 2), mtc::MAX_SPLIT));
  n = std::max(n, 1);
  int bps = (d.Kb + n - 1) / n;
  n = (d.Kb + bps - 1) / bps;
  if (n > mtc::MAX_SPLIT) return 0;
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
  if (n_split == 1)
    launch_pdl(attn_mla_tc_kernel, dim3(1, d.U, 2), dim3(mtc::THREADS), mtc::SMEM, s, d, L, q, sel, slot_of_sel, nsel,
               ctx_len, out, n_split, bps);
  else
    launch_pdl_cluster(attn_mla_tc_kernel, dim3(n_split, d.U, 2), dim3(mtc::THREADS), mtc::SMEM, s, (unsigned)n_split, d,
                       L, q, sel, slot_of_sel, nsel, ctx_len, out, n_split, bps);
  return cudaGetLastError();
}

}  // namespace kvs
