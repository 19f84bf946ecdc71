// Block-wide integer primitives: exclusive prefix sums and 8-bit-digit radix selection.
#pragma once
#include <stdint.h>

namespace kvs {

// Exclusive prefix sum over the CTA in thread order.  `ws` holds >= 33 ints of shared memory.
// Returns the exclusive prefix of v; *total receives the sum over the CTA.
__device__ __forceinline__ int block_excl_sum(int v, int* ws, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? ws[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) ws[lane] = w;          // inclusive warp totals
    if (lane == 31) ws[32] = w;
  }
  __syncthreads();
  int before = (warp > 0 ? ws[warp - 1] : 0) + x - v;
  *total = ws[32];
  __syncthreads();
  return before;
}

// One radix pass: given a 256-bin histogram `hist` (shared) of the current digit among the
// keys that still match the prefix, find the digit d holding the k-th key counted from the
// top (largest-first when `from_top`, else smallest-first).  Run by warp 0; results in
// out[0] = digit, out[1] = number of keys on the far side of d (strictly before it in the
// chosen order).
__device__ __forceinline__ void radix_pick_digit(const int* hist, int k, bool from_top, int* out) {
  const int lane = threadIdx.x & 31;
  // lane owns 8 bins in the chosen order: order position p = lane*8 + i
  int cnt[8];
  int local = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int p = lane * 8 + i;
    int bin = from_top ? 255 - p : p;
    cnt[i] = hist[bin];
    local += cnt[i];
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int excl = incl - local;
  if (excl < k && k <= incl) {
    int run = excl;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (run + cnt[i] >= k) {
        int p = lane * 8 + i;
        out[0] = from_top ? 255 - p : p;
        out[1] = run;
        break;
      }
      run += cnt[i];
    }
  }
}

}  // namespace kvs
