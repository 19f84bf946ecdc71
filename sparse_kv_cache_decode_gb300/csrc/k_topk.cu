// Block selection: forced sink/recent blocks plus the top (K_b - |forced|) other blocks by
// (score desc, block asc), emitted in ascending block order.
//
// Radix selection over orderable 32-bit keys (8-bit digits, most significant first) finds the
// threshold key T of the k-th best candidate and how many candidates equal to T are needed;
// an ordered compaction then takes every candidate above T and the lowest-index candidates
// equal to T: warp ballots over contiguous segments when the keys sit in shared memory
// (select_ordered), per-thread runs with block prefix sums when they are read from global memory.
// Contexts up to 16384 blocks: one CTA per unit.
//
// Long contexts (more blocks than one CTA caches in shared memory) select in two phases so that
// the work spreads over the SMs: (1) a grid of (chunk, unit) CTAs keeps, per chunk of 16384
// blocks, the chunk's own top-k candidates under the same order, in block order; (2) one CTA
// per unit selects the top-k among the kept candidates.  Every candidate of the unit's top-k is
// within the top-k of its own chunk (the candidates that precede it in the order are fewer
// than k), so the two phases select exactly the single-pass result.
#include "kvs_block.cuh"
#include "kvs_common.cuh"
#include "kvs_select.cuh"

namespace kvs {

namespace {

constexpr int kTopkThreads = 512;
constexpr int kTopkMaxChunks = 64;
constexpr size_t kTopkMergeSmemMax = 160 * 1024;  // kept candidates (key + block) of one unit

// The selection of unit u (nb blocks) with its keys read from the scores in global memory, for
// more blocks than shared memory holds: radix passes over the scores, then an ordered compaction
// (every thread of the CTA calls it).
__device__ void topk_unit_global(const Dims& d, const float* __restrict__ scores, int nb, int u, int* __restrict__ sel,
                                 int* __restrict__ nsel, unsigned* err, TopkShared& sh) {
  int* hist = sh.hist;
  int* ws = sh.ws;
  int* pick = sh.pick;
  const int tid = threadIdx.x, NT = blockDim.x;
  int* out = sel + (size_t)u * d.Kb;
  const float* s = scores + (size_t)u * d.nb_max;
  // more blocks than shared memory holds: the keys are read from the scores in global memory
  const int lo_forced = d.n_sink, hi_forced = nb - d.n_recent;  // forced: b < lo || b >= hi
  auto key_of = [&](int b) -> uint32_t { return score_key(s[b]); };
  auto is_cand = [&](int b) { return b >= lo_forced && b < hi_forced; };

  const int k = d.Kb - d.n_sink - d.n_recent;  // >= 0 checked at create
  uint32_t prefix = k > 0 ? 0u : 0xffffffffu;    // k == 0: no key reaches the threshold
  uint32_t mask = 0;
  int remaining = k;
  for (int pass = 0; pass < (k > 0 ? 4 : 0); ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += NT) hist[i] = 0;
    __syncthreads();
    for (int b = tid; b < nb; b += NT) {  // interleaved: coalesced reads
      if (!is_cand(b)) continue;
      uint32_t key = key_of(b);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid < 32) radix_pick_digit(hist, remaining, true, pick);
    __syncthreads();
    prefix |= (uint32_t)pick[0] << shift;
    mask |= 255u << shift;
    remaining -= pick[1];
    __syncthreads();
  }
  const uint32_t T = prefix;
  const int need_eq = remaining;

  // ordered compaction: thread t owns blocks [t*per, (t+1)*per)
  const int per = (nb + NT - 1) / NT;
  const int b0 = min(nb, tid * per), b1 = min(nb, b0 + per);
  int my_eq = 0;
  for (int b = b0; b < b1; ++b)
    if (is_cand(b) && key_of(b) == T) ++my_eq;
  int tot;
  int eq_rank = block_excl_sum(my_eq, ws, &tot);
  int my_take = 0;
  {
    int er = eq_rank;
    for (int b = b0; b < b1; ++b) {
      bool take;
      if (!is_cand(b)) take = true;
      else {
        uint32_t key = key_of(b);
        take = key > T || (key == T && er++ < need_eq);
      }
      my_take += take;
    }
  }
  int pos = block_excl_sum(my_take, ws, &tot);
  {
    int er = eq_rank;
    for (int b = b0; b < b1; ++b) {
      bool take;
      if (!is_cand(b)) take = true;
      else {
        uint32_t key = key_of(b);
        take = key > T || (key == T && er++ < need_eq);
      }
      if (take) {
        if (pos < d.Kb) out[pos] = b;
        ++pos;
      }
    }
  }
  if (tid == 0) {
    nsel[u] = tot;
    if (tot != d.Kb) set_error(err, KVS_ERR_BAD_INDEX);
  }
}


__global__ void __launch_bounds__(kTopkThreads) topk_kernel(Dims d, const float* __restrict__ scores,
                                                            const int* __restrict__ ctx_len, int* __restrict__ sel,
                                                            int* __restrict__ nsel, unsigned* err) {
  kvs_pdl_entry();
  extern __shared__ uint32_t skeys[];
  __shared__ TopkShared sh;
  const int u = blockIdx.x;
  const int r = u / d.Hkv;
  const int tid = threadIdx.x;
  const int len = ctx_len[r];
  if (len < 0 || len > d.max_ctx) {
    if (tid == 0) set_error(err, KVS_ERR_BAD_INDEX);
    return;
  }
  const int nb = n_blocks_of(len, d.bs);
  if (nb <= kTopkSmemKeys) {
    topk_unit_smem(d, scores, len, u, sel, nsel, err, skeys, sh);
    return;
  }
  topk_unit_global(d, scores, nb, u, sel, nsel, err, sh);
}

constexpr int kChunk = kTopkSmemKeys;   // blocks per phase-1 CTA
constexpr int kGuessSample = 4096;      // keys of the unit-wide threshold guess

// Whether a unit of `cand` candidate blocks (k to select) takes the unit-wide threshold guess.
__host__ __device__ inline bool use_unit_guess(int cand, int k) { return k > 0 && cand > 4 * k && cand > 4 * kGuessSample; }

// Unit-wide threshold guess T0: the key of rank about 1.25 k / cand of kGuessSample evenly spaced
// candidate keys (candidates are blocks [lo, lo + cand)).  Deterministic, so every chunk CTA of the
// unit and its merge CTA compute the same T0.  sample: kGuessSample words of shared memory.  Every
// thread of the CTA calls it.
__device__ uint32_t unit_guess(const float* __restrict__ s_unit, int lo, int cand, int k, uint32_t* sample,
                               TopkShared& sh, uint32_t* s_min) {
  const int tid = threadIdx.x, NT = blockDim.x;
  for (int i = tid; i < kGuessSample; i += NT) sample[i] = score_key(s_unit[lo + (long long)i * cand / kGuessSample]);
  if (tid == 0) *s_min = 0xffffffffu;
  __syncthreads();
  const int ks = min(kGuessSample, (int)(1.25f * (float)k * kGuessSample / (float)cand) + 16);
  // the ks-th largest sampled key = the smallest of the ks selected
  select_ordered(sample, kGuessSample, ks, sh.hist, sh.ws, sh.pick, [&](int, int i) { atomicMin(s_min, sample[i]); });
  const uint32_t t = *s_min;
  __syncthreads();
  return t;
}

// Phase 1: CTA (c, u) keeps candidates of blocks [c*kChunk, (c+1)*kChunk) of unit u (candidates:
// not sink, not recent), in block order, with their keys: for units that take the unit-wide
// threshold guess, the chunk's keys >= T0 (at most K_b of them; a chunk with more keeps its top-k,
// which is then a superset of its share of the answer whatever T0 is); otherwise the chunk's top-k.
__global__ void __launch_bounds__(kTopkThreads) topk_chunk_kernel(Dims d, const float* __restrict__ scores,
                                                                  const int* __restrict__ ctx_len, int P,
                                                                  uint32_t* __restrict__ ckey, int* __restrict__ cidx,
                                                                  int* __restrict__ ccnt) {
  kvs_pdl_entry();
  extern __shared__ uint32_t skeys[];                   // [kChunk] keys, then the threshold-guess scratch
  __shared__ TopkShared sh;
  __shared__ uint32_t s_min;
  __shared__ int s_cnt[33];
  const int c = blockIdx.x, u = blockIdx.y;
  const int tid = threadIdx.x, NT = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = NT >> 5;
  const int len = ctx_len[u / d.Hkv];
  const int nb = (len < 0 || len > d.max_ctx) ? 0 : n_blocks_of(len, d.bs);
  const int k = d.Kb - d.n_sink - d.n_recent;
  const size_t slot = (size_t)u * P + c;
  const int lo = d.n_sink, hi = nb - d.n_recent;
  const int b0 = max(c * kChunk, lo), b1 = min((c + 1) * kChunk, hi);
  const int n = (nb <= d.Kb || k <= 0) ? 0 : max(0, b1 - b0);
  const float* s = scores + (size_t)u * d.nb_max + b0;
  uint32_t* okey = ckey + slot * d.Kb;
  int* oidx = cidx + slot * d.Kb;
  const bool guess = nb > d.Kb && use_unit_guess(hi - lo, k);
  uint32_t T0 = 0u;
  if (guess) T0 = unit_guess(scores + (size_t)u * d.nb_max, lo, hi - lo, k, skeys + kChunk, sh, &s_min);
  if (!guess && n <= k) {                              // every candidate of the chunk is kept
    for (int i = tid; i < n; i += NT) {
      okey[i] = score_key(s[i]);
      oidx[i] = b0 + i;
    }
    if (tid == 0) ccnt[slot] = n;
    return;
  }
  for (int i = tid; i < n; i += NT) skeys[i] = score_key(s[i]);
  __syncthreads();
  if (guess) {
    // keys >= T0, counted per warp segment, then compacted in block order
    const int seg = ((n + nw - 1) / nw + 31) & ~31;
    const int w0 = min(n, warp * seg), w1 = min(n, w0 + seg);
    int cw = 0;
    for (int base = w0; base < w1; base += 32) {
      const int i = base + lane;
      cw += __popc(__ballot_sync(0xffffffffu, i < w1 && skeys[i] >= T0));
    }
    if (lane == 0) s_cnt[warp] = cw;
    __syncthreads();
    int total = 0, off = 0;
    for (int w = 0; w < nw; ++w) {
      if (w < warp) off += s_cnt[w];
      total += s_cnt[w];
    }
    if (total <= d.Kb) {
      const unsigned below = (1u << lane) - 1u;
      for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const bool p = i < w1 && skeys[i] >= T0;
        const unsigned m = __ballot_sync(0xffffffffu, p);
        if (p) {
          okey[off + __popc(m & below)] = skeys[i];
          oidx[off + __popc(m & below)] = b0 + i;
        }
        off += __popc(m);
      }
      if (tid == 0) ccnt[slot] = total;
      return;
    }
    __syncthreads();                                   // s_cnt and the scratch are free again
  }
  select_topk(skeys, n, k, skeys + kChunk, sh, [&](int r, int i) {
    okey[r] = skeys[i];
    oidx[r] = b0 + i;
  });
  if (tid == 0) ccnt[slot] = k;
}

// Phase 2: one CTA per unit selects the top-k among its chunks' kept candidates and frames them
// with the sink and recent blocks, in ascending block order.
__global__ void __launch_bounds__(kTopkThreads) topk_merge_kernel(Dims d, const float* __restrict__ scores,
                                                                  const int* __restrict__ ctx_len, int P,
                                                                  const uint32_t* __restrict__ ckey,
                                                                  const int* __restrict__ cidx,
                                                                  const int* __restrict__ ccnt, int* __restrict__ sel,
                                                                  int* __restrict__ nsel, unsigned* err) {
  kvs_pdl_entry();
  extern __shared__ uint32_t smem[];                    // [P * Kb] keys, [P * Kb] blocks, guess scratch
  __shared__ TopkShared sh;
  __shared__ int off[kTopkMaxChunks + 1];
  __shared__ uint32_t s_min;
  __shared__ int s_ge;
  const int u = blockIdx.x;
  const int tid = threadIdx.x, NT = blockDim.x;
  const int len = ctx_len[u / d.Hkv];
  if (len < 0 || len > d.max_ctx) {
    if (tid == 0) set_error(err, KVS_ERR_BAD_INDEX);
    return;
  }
  const int nb = n_blocks_of(len, d.bs);
  int* out = sel + (size_t)u * d.Kb;
  if (nb <= d.Kb) {
    for (int i = tid; i < nb; i += NT) out[i] = i;
    if (tid == 0) nsel[u] = nb;
    return;
  }
  const int k = d.Kb - d.n_sink - d.n_recent;
  for (int i = tid; i < d.n_sink; i += NT) out[i] = i;
  for (int i = tid; i < d.n_recent; i += NT) out[d.n_sink + k + i] = nb - d.n_recent + i;
  if (tid == 0) {
    int o = 0;
    for (int c = 0; c < P; ++c) {
      off[c] = o;
      o += ccnt[(size_t)u * P + c];
    }
    off[P] = o;
  }
  __syncthreads();
  const int n = off[P];
  uint32_t* keys = smem;
  int* idx = reinterpret_cast<int*>(smem + (size_t)P * d.Kb);
  for (int c = 0; c < P; ++c) {
    const size_t slot = (size_t)u * P + c;
    const int m = off[c + 1] - off[c];
    for (int i = tid; i < m; i += NT) {
      keys[off[c] + i] = ckey[slot * d.Kb + i];
      idx[off[c] + i] = cidx[slot * d.Kb + i];
    }
  }
  __syncthreads();
  if (k > 0 && use_unit_guess(nb - d.n_recent - d.n_sink, k)) {
    // the chunks kept keys >= T0 (or their top-k): the kept lists hold the answer when at least k
    // kept keys are >= T0 (the k-th largest key is then >= T0); else the unit is selected again
    // from its scores in global memory
    uint32_t* scratch = smem + (size_t)2 * P * d.Kb;
    const uint32_t T0 = unit_guess(scores + (size_t)u * d.nb_max, d.n_sink, nb - d.n_recent - d.n_sink, k, scratch, sh,
                                   &s_min);
    if (tid == 0) s_ge = 0;
    __syncthreads();
    int ge = 0;
    for (int i = tid; i < n; i += NT) ge += keys[i] >= T0;
    if (ge) atomicAdd(&s_ge, ge);
    __syncthreads();
    if (s_ge < k) {
      topk_unit_global(d, scores, nb, u, sel, nsel, err, sh);
      return;
    }
  }
  if (k > 0) {
    // nb > Kb leaves more than k candidates, so at least k were kept; exactly k when a single
    // chunk held more than k of them (all kept ones are then the answer)
    if (n < k) {
      if (tid == 0) set_error(err, KVS_ERR_BAD_INDEX);
      return;
    }
    if (n == k) {
      for (int i = tid; i < n; i += NT) out[d.n_sink + i] = idx[i];
    } else {
      select_topk(keys, n, k, smem + (size_t)2 * P * d.Kb, sh, [&](int r, int i) { out[d.n_sink + r] = idx[i]; });
    }
  }
  if (tid == 0) nsel[u] = d.Kb;
}

}  // namespace

int topk_chunks(const Dims& d) {
  if (d.nb_max <= kTopkSmemKeys) return 0;
  const int P = (d.nb_max + kChunk - 1) / kChunk;
  const size_t merge_smem = (size_t)P * d.Kb * 8;
  if (P > kTopkMaxChunks || merge_smem > kTopkMergeSmemMax) return 0;   // single pass
  return P;
}

cudaError_t launch_topk(const Dims& d, const float* scores, const int* ctx_len, int* sel, int* nsel, unsigned* err,
                        cudaStream_t s, const TopkScratch* scratch) {
  const int P = scratch ? topk_chunks(d) : 0;
  if (P > 0) {
    // each kernel's keys plus the scratch of the threshold guess (kTopkFastScratch words)
    const size_t chunk_smem = (kChunk + kTopkFastScratch) * sizeof(uint32_t);
    const size_t merge_smem = (size_t)P * d.Kb * 8 + kTopkFastScratch * sizeof(uint32_t);
    {
      cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(topk_chunk_kernel), (int)chunk_smem);
      if (e == cudaSuccess) e = set_max_dynamic_smem(reinterpret_cast<const void*>(topk_merge_kernel), (int)merge_smem);
      if (e != cudaSuccess) return e;
    }
    launch_pdl(topk_chunk_kernel, dim3(dim3(P, d.U)), dim3(kTopkThreads), chunk_smem, s, d, scores, ctx_len, P,
               scratch->key, scratch->idx, scratch->cnt);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    launch_pdl(topk_merge_kernel, dim3(d.U), dim3(kTopkThreads), merge_smem, s, d, scores, ctx_len, P, scratch->key,
               scratch->idx, scratch->cnt, sel, nsel, err);
    return cudaGetLastError();
  }
  size_t smem = (size_t)kTopkSmemKeys * sizeof(uint32_t);
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(topk_kernel), (int)smem);
    if (e != cudaSuccess) return e;
  }
  launch_pdl(topk_kernel, dim3(d.U), dim3(kTopkThreads), smem, s, d, scores, ctx_len, sel, nsel, err);
  return cudaGetLastError();
}

}  // namespace kvs
