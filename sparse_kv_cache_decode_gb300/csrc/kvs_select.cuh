// Block selection in shared memory (one CTA per unit): the radix top-k over orderable 32-bit
// keys shared by the top-K kernels and the fused top-K + cache update kernel.
#pragma once
#include "kvs_block.cuh"
#include "kvs_common.cuh"
#include "kvs_ptx.cuh"

namespace kvs {

constexpr int kTopkSmemKeys = 16384;   // block scores a CTA caches in shared memory (one unit)

// Histogram of one 8-bit digit over the keys in shared memory that match `prefix` under
// `mask`.  The lanes of a warp that hold the same digit add their count once (the keys of one
// unit share their high bytes, so on the first passes most keys land in one or two bins).
__device__ __forceinline__ void digit_histogram(const uint32_t* keys, int n, uint32_t prefix, uint32_t mask,
                                                int shift, int* hist) {
  const int lane = threadIdx.x & 31;
  for (int base = threadIdx.x - lane; base < n; base += blockDim.x) {   // warp-uniform trip count
    const int i = base + lane;
    int bin = -1;
    if (i < n) {
      const uint32_t key = keys[i];
      if ((key & mask) == prefix) bin = (int)((key >> shift) & 255u);
    }
    const unsigned peers = __match_any_sync(0xffffffffu, bin);
    if (bin >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
  }
}

// Top k of keys[0, n) in shared memory by (key desc, position asc); emit(rank, i) is called for
// each selected position i, ranks 0..k-1 in ascending position order.  Every thread of the CTA
// (at most 512) must call it.  Requires 0 < k < n.  ws holds at least 33 ints.
//
// The threshold key T and the number of keys equal to T still needed come from 8-bit radix passes
// (at most four), cut short once at most 32 keys still match the prefix.  The compaction gives
// each warp a contiguous segment of positions and walks it 32 keys at a time (lane i reads
// position base + i: no bank conflicts); ballots give each lane its rank among the equal keys and
// among the taken keys.
template <class Emit>
__device__ void select_ordered(const uint32_t* keys, int n, int k, int* hist, int* ws, int* pick, Emit emit) {
  const int tid = threadIdx.x, NT = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = NT >> 5;
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  if (tid == 0) ws[32] = 0;   // gather counter of the short finish (below)
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += NT) hist[i] = 0;
    __syncthreads();
    digit_histogram(keys, n, prefix, mask, shift, hist);
    __syncthreads();
    if (tid < 32) radix_pick_digit(hist, remaining, true, pick);
    __syncthreads();
    prefix |= (uint32_t)pick[0] << shift;
    mask |= 255u << shift;
    remaining -= pick[1];
    const int in_bin = hist[pick[0]];   // keys that match the longer prefix
    __syncthreads();
    if (pass < 3 && in_bin <= 32) {
      // Short finish: the threshold is the remaining-th largest of the <= 32 keys that match the
      // prefix.  They are gathered (in any order) into the free histogram, and one warp finds it
      // by counting, for each key, the keys above it and equal to it.
      for (int i = tid; i < n; i += NT) {
        const uint32_t key = keys[i];
        if ((key & mask) == prefix) hist[atomicAdd(&ws[32], 1)] = (int)key;
      }
      __syncthreads();
      if (warp == 0) {
        const int cnt = ws[32];
        const uint32_t mine = lane < cnt ? (uint32_t)hist[lane] : 0u;
        int gt = 0, eq = 0;
        for (int j = 0; j < cnt; ++j) {
          const uint32_t kj = (uint32_t)__shfl_sync(0xffffffffu, (int)mine, j);
          gt += kj > mine;
          eq += kj == mine;
        }
        const bool is_t = lane < cnt && gt < remaining && remaining <= gt + eq;
        const int src = __ffs(__ballot_sync(0xffffffffu, is_t)) - 1;   // some lane holds the threshold
        const int t_gt = __shfl_sync(0xffffffffu, gt, src);
        const uint32_t t_key = (uint32_t)__shfl_sync(0xffffffffu, (int)mine, src);
        if (lane == 0) {
          pick[0] = (int)t_key;
          pick[1] = remaining - t_gt;
        }
      }
      __syncthreads();
      prefix = (uint32_t)pick[0];
      remaining = pick[1];
      __syncthreads();   // pick and hist are free again
      break;
    }
  }
  const uint32_t T = prefix;
  const int need_eq = remaining;
  const int seg = ((n + nw - 1) / nw + 31) & ~31;
  const int w0 = min(n, warp * seg), w1 = min(n, w0 + seg);
  int c_eq = 0, c_gt = 0;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < w1 ? keys[i] : 0u;
    c_eq += __popc(__ballot_sync(0xffffffffu, i < w1 && key == T));
    c_gt += __popc(__ballot_sync(0xffffffffu, i < w1 && key > T));
  }
  if (lane == 0) {
    ws[warp] = c_eq;
    ws[16 + warp] = c_gt;
  }
  __syncthreads();
  int run_eq = 0, run_take = 0;
  for (int w = 0; w < warp; ++w) {
    const int e = ws[w];
    run_take += ws[16 + w] + max(0, min(e, need_eq - run_eq));
    run_eq += e;
  }
  const unsigned below = (1u << lane) - 1u;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < w1 ? keys[i] : 0u;
    const bool eq = i < w1 && key == T;
    const unsigned eqm = __ballot_sync(0xffffffffu, eq);
    const bool take = (i < w1 && key > T) || (eq && run_eq + __popc(eqm & below) < need_eq);
    const unsigned tm = __ballot_sync(0xffffffffu, take);
    if (take) emit(run_take + __popc(tm & below), i);
    run_eq += __popc(eqm);
    run_take += __popc(tm);
  }
  __syncthreads();
}


struct TopkShared {
  int hist[256];
  int ws[33];
  int pick[2];
};

constexpr int kTopkSample = 256;       // sampled keys of the threshold guess
constexpr int kTopkFastMax = 4096;     // keys at or above the guess kept for the exact selection
constexpr int kTopkFastScratch = kTopkSample + 2 * kTopkFastMax;   // 32-bit words of shared scratch

// select_ordered, fronted by a threshold guess when the keys are many: T0 = a sampled key of rank
// about 1.25 k n / 256 among 256 evenly spaced keys; if between k and kTopkFastMax keys are >= T0,
// they (with their positions, in position order) are the only candidates: every selected key and
// every key equal to the k-th largest is >= T0, so the exact selection among them is the same.
// Otherwise the full selection runs.  scratch: kTopkFastScratch words of shared memory, or null
// (always the full selection).  Same contract as select_ordered.
template <class Emit>
__device__ void select_topk(const uint32_t* keys, int n, int k, uint32_t* scratch, TopkShared& sh, Emit emit) {
  const int tid = threadIdx.x, NT = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = NT >> 5;
  if (scratch == nullptr || n < 4 * k || n <= 2 * kTopkSample) {
    select_ordered(keys, n, k, sh.hist, sh.ws, sh.pick, emit);
    return;
  }
  uint32_t* sample = scratch;
  uint32_t* lkey = scratch + kTopkSample;
  int* lpos = reinterpret_cast<int*>(lkey + kTopkFastMax);
  for (int i = tid; i < kTopkSample; i += NT) sample[i] = keys[(long long)i * n / kTopkSample];
  const int ks = min(kTopkSample, (int)(1.25f * (float)k * kTopkSample / (float)n) + 8);
  if (tid == 0) sh.ws[32] = 0;
  __syncthreads();
  // the ks-th largest sampled key (ties by sample index)
  for (int i = tid; i < kTopkSample; i += NT) {
    const uint32_t v = sample[i];
    int r = 0;
    for (int j = 0; j < kTopkSample; ++j) {
      const uint32_t sj = sample[j];
      r += sj > v || (sj == v && j < i);
    }
    if (r == ks - 1) sh.pick[0] = (int)v;
  }
  __syncthreads();
  const uint32_t T0 = (uint32_t)sh.pick[0];
  // keys >= T0, counted a warp at a time
  const int seg = ((n + nw - 1) / nw + 31) & ~31;
  const int w0 = min(n, warp * seg), w1 = min(n, w0 + seg);
  int cw = 0;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    cw += __popc(__ballot_sync(0xffffffffu, i < w1 && keys[i] >= T0));
  }
  if (lane == 0) {
    sh.ws[warp] = cw;
    atomicAdd(&sh.ws[32], cw);
  }
  __syncthreads();
  const int cnt = sh.ws[32];
  if (cnt < k || cnt > kTopkFastMax) {
    __syncthreads();
    select_ordered(keys, n, k, sh.hist, sh.ws, sh.pick, emit);
    return;
  }
  // ordered compaction of the keys >= T0 (warp segments in order, ballots within a segment)
  int off = 0;
  for (int w = 0; w < warp; ++w) off += sh.ws[w];
  const unsigned below = (1u << lane) - 1u;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < w1 ? keys[i] : 0u;
    const bool p = i < w1 && key >= T0;
    const unsigned m = __ballot_sync(0xffffffffu, p);
    if (p) {
      lkey[off + __popc(m & below)] = key;
      lpos[off + __popc(m & below)] = i;
    }
    off += __popc(m);
  }
  __syncthreads();
  if (cnt == k) {
    for (int i = tid; i < cnt; i += NT) emit(i, lpos[i]);
    __syncthreads();
    return;
  }
  select_ordered(lkey, cnt, k, sh.hist, sh.ws, sh.pick, [&](int r, int i) { emit(r, lpos[i]); });
}

// Selection of unit u from its block scores when the unit's candidates fit the `skeys` shared
// buffer: forced sink and recent blocks plus the top (K_b - forced) other blocks by (score desc,
// block asc), in ascending block order, into sel[u][..] and nsel[u].  In two phases, so that the
// score reads can travel with other reads of the caller:
//   topk_stage issues the reads of the unit's score row (blocks [0, nb - n_recent)) into skeys,
//   through L2 (the scores may have been written by other CTAs of the running kernel);
//   after cp_async_wait_all and a CTA barrier, topk_staged turns them into orderable keys in
//   place and selects; it returns the selection's count (also copied to out_s when not null), or
//   -1 for a context length out of range (KVS_ERR_BAD_INDEX, nothing written); fast_scratch
//   (kTopkFastScratch words of shared memory, or null) enables select_topk's threshold guess.
// Every thread of the CTA calls both.
__device__ inline void topk_stage(const Dims& d, const float* scores, int len, int u, uint32_t* skeys) {
  if (len < 0 || len > d.max_ctx) return;
  const int nb = n_blocks_of(len, d.bs);
  if (nb <= d.Kb) return;
  const int n_stage = min(d.nb_max, (nb - d.n_recent + 3) & ~3);
  stage_words(skeys, scores + (size_t)u * d.nb_max, n_stage);
}

__device__ inline int topk_staged(const Dims& d, int len, int u, int* __restrict__ sel, int* __restrict__ nsel,
                                  unsigned* err, uint32_t* skeys, int* out_s, TopkShared& sh,
                                  uint32_t* fast_scratch = nullptr) {
  const int tid = threadIdx.x, NT = blockDim.x;
  if (len < 0 || len > d.max_ctx) {
    if (tid == 0) set_error(err, KVS_ERR_BAD_INDEX);
    return -1;
  }
  const int nb = n_blocks_of(len, d.bs);
  int* out = sel + (size_t)u * d.Kb;
  if (nb <= d.Kb) {
    for (int i = tid; i < nb; i += NT) {
      out[i] = i;
      if (out_s) out_s[i] = i;
    }
    if (tid == 0) nsel[u] = nb;
    return nb;
  }
  const int lo_forced = d.n_sink, hi_forced = nb - d.n_recent;  // forced: b < lo || b >= hi
  const int k_free = d.Kb - d.n_sink - d.n_recent;              // >= 0 checked at create
  // candidates [lo_forced, hi_forced) are contiguous: their keys, in place (each thread converts
  // the words it reads); the result is framed with the forced blocks (sinks first, recent last)
  for (int b = lo_forced + tid; b < hi_forced; b += NT) skeys[b] = score_key(__uint_as_float(skeys[b]));
  for (int i = tid; i < d.n_sink; i += NT) {
    out[i] = i;
    if (out_s) out_s[i] = i;
  }
  for (int i = tid; i < d.n_recent; i += NT) {
    out[d.n_sink + k_free + i] = hi_forced + i;
    if (out_s) out_s[d.n_sink + k_free + i] = hi_forced + i;
  }
  __syncthreads();
  if (k_free > 0)
    select_topk(skeys + lo_forced, hi_forced - lo_forced, k_free, fast_scratch, sh, [&](int r, int i) {
      out[d.n_sink + r] = lo_forced + i;
      if (out_s) out_s[d.n_sink + r] = lo_forced + i;
    });
  if (tid == 0) nsel[u] = d.Kb;
  return d.Kb;
}

// Both phases back to back (the score reads alone in their round).
__device__ inline void topk_unit_smem(const Dims& d, const float* scores, int len, int u, int* __restrict__ sel,
                                      int* __restrict__ nsel, unsigned* err, uint32_t* skeys, TopkShared& sh) {
  topk_stage(d, scores, len, u, skeys);
  cp_async_wait_all();
  __syncthreads();
  topk_staged(d, len, u, sel, nsel, err, skeys, nullptr, sh);
}

}  // namespace kvs
