// Block selection: forced sink/recent blocks plus the top (K_b - |forced|) other blocks by
// (score desc, block asc), emitted in ascending block order.  One CTA per unit.
//
// Radix selection over orderable 32-bit keys (8-bit digits, most significant first) finds the
// threshold key T of the k-th best candidate and how many candidates equal to T are needed;
// an ordered compaction (prefix sums in block order) then takes every candidate above T and
// the lowest-index candidates equal to T.
#include "kvs_block.cuh"
#include "kvs_common.cuh"

namespace kvs {

namespace {

constexpr int kTopkThreads = 512;
constexpr int kTopkSmemKeys = 16384;  // scores cached in shared memory up to this many blocks

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(Dims d, const float* __restrict__ scores,
                                                            const int* __restrict__ ctx_len, int* __restrict__ sel,
                                                            int* __restrict__ nsel, unsigned* err) {
  extern __shared__ uint32_t skeys[];
  __shared__ int hist[256];
  __shared__ int ws[33];
  __shared__ int pick[2];
  const int u = blockIdx.x;
  const int r = u / d.Hkv;
  const int tid = threadIdx.x, NT = blockDim.x;
  const int len = ctx_len[r];
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
  const float* s = scores + (size_t)u * d.nb_max;
  const int lo_forced = d.n_sink, hi_forced = nb - d.n_recent;  // forced: b < lo || b >= hi
  const bool cached = nb <= kTopkSmemKeys;
  if (cached) {
    for (int i = tid; i < nb; i += NT) skeys[i] = score_key(s[i]);
    __syncthreads();
  }
  auto key_of = [&](int b) -> uint32_t { return cached ? skeys[b] : score_key(s[b]); };
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

}  // namespace

cudaError_t launch_topk(const Dims& d, const float* scores, const int* ctx_len, int* sel, int* nsel, unsigned* err,
                        cudaStream_t s) {
  size_t smem = (size_t)kTopkSmemKeys * sizeof(uint32_t);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  topk_kernel<<<d.U, kTopkThreads, smem, s>>>(d, scores, ctx_len, sel, nsel, err);
  return cudaGetLastError();
}

}  // namespace kvs
