// GPU working-set cache of each (request, layer, kv-head) unit: the update kernels (the update body
// itself is in kvs_update.cuh; one CTA per unit, so the state of a unit has a single writer), the
// cross-layer prefetch, the snapshot restore, and the zero-copy host -> slot fetch of the blocks
// each of them maps.
#include "kvs_block.cuh"
#include "kvs_common.cuh"
#include "kvs_ptx.cuh"
#include "kvs_select.cuh"
#include "kvs_update.cuh"

#include <algorithm>

namespace kvs {

namespace {

__global__ void __launch_bounds__(kCacheThreads) cache_update_kernel(Dims d, Layer L, const int* __restrict__ sel,
                                                                     const int* __restrict__ nsel,
                                                                     const int* __restrict__ ctx_len,
                                                                     int* __restrict__ slot_of_sel,
                                                                     const float* __restrict__ imp, kvs_stats* stats) {
  kvs_pdl_entry();
  extern __shared__ __align__(16) unsigned char smraw[];
  __shared__ UpdateShared sh;
  update_unit(d, L, blockIdx.x, sel, nsel, ctx_len, slot_of_sel, imp, stats, smraw, sh);
}

// Top-K selection and cache update of one unit in one CTA (contexts of at most kTopkSmemKeys
// blocks): the selection goes to sel / nsel as from the top-K kernel and, through shared memory,
// to the update, with no kernel boundary between the two.
__global__ void __launch_bounds__(kCacheThreads) select_update_kernel(Dims d, Layer L, const float* __restrict__ scores,
                                                                      const int* __restrict__ ctx_len, int* sel,
                                                                      int* nsel, int* __restrict__ slot_of_sel,
                                                                      kvs_stats* stats) {
  kvs_pdl_entry();
  extern __shared__ __align__(16) unsigned char smraw[];
  __shared__ TopkShared tsh;
  __shared__ UpdateShared ush;
  const int u = blockIdx.x;
  // one round of reads: the score row and every update input that does not depend on the selection
  UpdateIn in = update_stage(d, L, u, ctx_len, smraw, ush);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smraw + select_keys_offset(d));
  topk_stage(d, scores, in.len, u, keys);
  cp_async_wait_all();
  __syncthreads();
  in.n = topk_staged(d, in.len, u, sel, nsel, L.err, keys, update_sel_buffer(d, smraw), tsh,
                     reinterpret_cast<uint32_t*>(smraw + select_scratch_offset(d)));
  __syncthreads();
  update_run(d, L, u, in, slot_of_sel, d.evict_importance ? scores : nullptr, stats, smraw, ush);
}

__global__ void __launch_bounds__(kCacheThreads) prefetch_kernel(Dims d, Layer L, const int* __restrict__ hint,
                                                                 const int* __restrict__ hint_n,
                                                                 const int* __restrict__ ctx_len, kvs_stats* stats) {
  kvs_pdl_entry();
  extern __shared__ __align__(16) unsigned char smraw[];
  __shared__ int hist[256];
  __shared__ int ws[33];
  __shared__ int pick[2];
  __shared__ int s_bad;
  __shared__ unsigned long long s_cnt[2];  // evictions, bytes
  CacheSmem sm = carve(smraw, d);
  const int u = blockIdx.x, r = u / d.Hkv;
  const int tid = threadIdx.x, NT = blockDim.x;
  const int len = ctx_len[r];
  const int nh = hint_n[u];
  const int nb = n_blocks_of(len, d.bs);
  if (len < 0 || len > d.max_ctx || nh < 0 || nh > d.Kb) {
    if (tid == 0) {
      set_error(L.err, KVS_ERR_BAD_INDEX);
      L.n_fetch[u] = 0;
    }
    return;
  }
  const int* hu = hint + (size_t)u * d.Kb;
  int* b2s = L.block2slot + (size_t)u * d.nb_max;
  int* s2b = L.slot2block + (size_t)u * d.C;
  unsigned* st = L.stamp + (size_t)u * d.C;
  const unsigned clk = L.clock[u];
  const unsigned tag = 2u * clk + 1u, last_use = 2u * clk;
  if (tid == 0) s_bad = 0;
  if (tid < 2) s_cnt[tid] = 0;
  for (int s = tid; s < d.C; s += NT) sm.flags[s] = 0;
  __syncthreads();
  const int per = (nh + NT - 1) / NT;
  const int i0 = min(nh, tid * per), i1 = min(nh, i0 + per);
  int my_nr = 0;
  for (int i = i0; i < i1; ++i) {
    int b = hu[i];
    if (b < 0 || b >= nb || (i > 0 && hu[i - 1] >= b)) { s_bad = 1; continue; }
    int s = b2s[b];
    if (s >= d.C) { s_bad = 1; continue; }
    if (s >= 0) sm.flags[s] = 1; else ++my_nr;
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      set_error(L.err, KVS_ERR_BAD_INDEX);
      L.n_fetch[u] = 0;
    }
    return;
  }
  int n_nr;
  int pos = block_excl_sum(my_nr, ws, &n_nr);
  for (int i = i0; i < i1; ++i) {
    int b = hu[i];
    if (b2s[b] < 0) sm.list_blk[pos++] = b;
  }
  auto elig = [&](int s) { return s2b[s] < 0 || (st[s] < last_use && sm.flags[s] == 0); };
  int my_el = 0;
  for (int s = tid; s < d.C; s += NT) my_el += elig(s);
  int n_el;
  block_excl_sum(my_el, ws, &n_el);
  const int k = min(min(n_nr, d.max_prefetch), n_el);
  select_victims(d.C, k, elig, [&](int s) { return s2b[s] < 0 ? 0u : st[s]; }, hist, ws, pick, sm);
  unsigned long long my_ev = 0, my_bytes = 0;
  for (int j = tid; j < k; j += NT) {
    int b = sm.list_blk[j], s = sm.vict[j];
    int old = s2b[s];
    if (old >= 0 && old < d.nb_max) { b2s[old] = -1; ++my_ev; }
    s2b[s] = b;
    b2s[b] = s;
    st[s] = tag;
    L.fetch_blk[(size_t)u * d.C + j] = b;
    L.fetch_slot[(size_t)u * d.C + j] = s;
    my_bytes += fetch_rows(d, len, b) * (unsigned long long)d.row_bytes;
  }
  if (my_ev) atomicAdd(&s_cnt[0], my_ev);
  if (my_bytes) atomicAdd(&s_cnt[1], my_bytes);
  __syncthreads();
  if (tid == 0) {
    L.n_fetch[u] = k;
    if (stats) {
      kvs_stats* sl = stats + L.layer;
      atomicAdd(&sl->prefetched, (unsigned long long)k);
      atomicAdd(&sl->evictions, s_cnt[0]);
      atomicAdd(&sl->bytes_fetched, s_cnt[1]);
    }
  }
}

// Restore of one unit from a snapshot (one CTA per unit): the slots whose block differs from the
// snapshot's (where the snapshot's slot held a block) go to the unit's fetch list in slot order,
// then the snapshot's maps, stamps, clock and pending selection are copied back.  A snapshot
// block id outside [-1, n_b(max_ctx)) is reported (KVS_ERR_BAD_INDEX) and not fetched.
constexpr int kRestoreThreads = 256;

__global__ void __launch_bounds__(kRestoreThreads) restore_kernel(Dims d, Layer L, const unsigned char* __restrict__ snap,
                                                                  SnapshotPlan p) {
  kvs_pdl_entry();
  __shared__ int ws[33];
  const int u = blockIdx.x, tid = threadIdx.x, NT = blockDim.x;
  const int* sb2s = reinterpret_cast<const int*>(snap) + (size_t)u * d.nb_max;
  const int* ss2b = reinterpret_cast<const int*>(snap + p.b2s) + (size_t)u * d.C;
  const unsigned* sst = reinterpret_cast<const unsigned*>(snap + p.b2s + p.s2b) + (size_t)u * d.C;
  const unsigned* sclk = reinterpret_cast<const unsigned*>(snap + p.b2s + p.s2b + p.stamp);
  const int* spsel = reinterpret_cast<const int*>(snap + p.b2s + p.s2b + p.stamp + p.clock) + (size_t)u * d.Kb;
  const int* spslot =
      reinterpret_cast<const int*>(snap + p.b2s + p.s2b + p.stamp + p.clock + p.pend_sel) + (size_t)u * d.Kb;
  const int* spn = reinterpret_cast<const int*>(snap + p.b2s + p.s2b + p.stamp + p.clock + p.pend_sel + p.pend_slot);
  int* b2s = L.block2slot + (size_t)u * d.nb_max;
  int* s2b = L.slot2block + (size_t)u * d.C;
  unsigned* st = L.stamp + (size_t)u * d.C;
  const int per = (d.C + NT - 1) / NT;
  const int s0 = min(d.C, tid * per), s1 = min(d.C, s0 + per);
  auto needs = [&](int s) {
    const int want = ss2b[s];
    if (want < -1 || want >= d.nb_max) {
      set_error(L.err, KVS_ERR_BAD_INDEX);
      return false;
    }
    return want >= 0 && s2b[s] != want;
  };
  int mine = 0;
  for (int s = s0; s < s1; ++s) mine += needs(s);
  int total;
  int pos = block_excl_sum(mine, ws, &total);
  for (int s = s0; s < s1; ++s) {
    if (!needs(s)) continue;
    L.fetch_blk[(size_t)u * d.C + pos] = ss2b[s];
    L.fetch_slot[(size_t)u * d.C + pos] = s;
    ++pos;
  }
  __syncthreads();   // every read of the live slot map is done before it is overwritten
  for (int i = tid; i < d.nb_max; i += NT) b2s[i] = sb2s[i];
  for (int s = tid; s < d.C; s += NT) {
    s2b[s] = ss2b[s];
    st[s] = sst[s];
  }
  for (int i = tid; i < d.Kb; i += NT) {
    L.pend_sel[(size_t)u * d.Kb + i] = spsel[i];
    L.pend_slot[(size_t)u * d.Kb + i] = spslot[i];
  }
  if (tid == 0) {
    L.clock[u] = sclk[u];
    L.pend_n[u] = spn[u];
    L.next_commit[u] = 0;
    L.n_fetch[u] = total;
  }
}

// Zero-copy fetch with one small CTA per SM, so that it fits beside the compute kernels that run
// with it, and a layer's misses are all in flight at once (the host link needs a few MB in flight
// to reach its peak): the CTAs flatten the (unit, item) lists with a prefix sum over units; each
// warp copies batches of whole items (about 512 16-byte vectors per batch), 16 loads in flight
// per lane, from the mapped host history into the items' slots.  Only rows < L are copied.
constexpr int kFetchThreads = 128;   // about 12K registers per CTA (one item per batch): fits beside two attention CTAs
constexpr int kFetchMaxUnits = 1024;
constexpr int kFetchUnroll = 16;

// Items per warp batch: whole items of about 512 16-byte vectors.
__host__ __device__ inline int fetch_items_per_batch(const Dims& d) {
  const int vpi = d.bs * d.dk * d.ebytes / 16 + (d.v_shares_k ? 0 : d.bs * d.dv * d.ebytes / 16);
  return vpi >= 512 ? 1 : 512 / vpi;
}

// SINGLE: one item per warp batch (items of 512 vectors or more); every lane locates the item
// itself, so no per-vector item state is held (a small register footprint).
template <bool SINGLE>
__global__ void __launch_bounds__(kFetchThreads, SINGLE ? 5 : 1) fetch_kernel(Dims d, Layer L, const int* __restrict__ ctx_len) {
  kvs_pdl_entry();
  __shared__ int s_off[kFetchMaxUnits + 1];
  __shared__ int ws[33];
  const int tid = threadIdx.x, lane = tid & 31;
  // prefix sum of the per-unit item counts
  const int per = (d.U + blockDim.x - 1) / blockDim.x;
  const int u0 = min(d.U, tid * per), u1 = min(d.U, u0 + per);
  int mine = 0;
  for (int u = u0; u < u1; ++u) mine += L.n_fetch[u];
  int total;
  int off = block_excl_sum(mine, ws, &total);
  for (int u = u0; u < u1; ++u) { s_off[u] = off; off += L.n_fetch[u]; }
  if (tid == 0) s_off[d.U] = total;
  __syncthreads();

  const int kvec = d.dk * d.ebytes / 16, vvec = d.dv * d.ebytes / 16;   // 16-byte vectors of a K / V row
  const int vk = d.bs * kvec;                             // of K in a full block
  const int vv = d.v_shares_k ? 0 : d.bs * vvec;
  const int vpi = vk + vv;
  const int ipb = fetch_items_per_batch(d);
  const int n_batches = (total + ipb - 1) / ipb;
  const int gwarp = blockIdx.x * (blockDim.x >> 5) + (tid >> 5);
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  if (SINGLE) {
    for (int item = gwarp; item < total; item += nwarps) {
      int lo = 0, hi = d.U;                               // s_off[lo] <= item < s_off[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= item) lo = mid; else hi = mid;
      }
      const int j = item - s_off[lo];
      const int b = L.fetch_blk[(size_t)lo * d.C + j], sl = L.fetch_slot[(size_t)lo * d.C + j];
      const int rows = max(0, min(d.bs, ctx_len[lo / d.Hkv] - b * d.bs));
      const size_t src_row = (size_t)lo * d.max_ctx + (size_t)b * d.bs, dst_row = ((size_t)lo * d.C + sl) * d.bs;
      const uint4* ks = reinterpret_cast<const uint4*>(L.host_k) + src_row * kvec;
      const uint4* vs = reinterpret_cast<const uint4*>(L.host_v) + src_row * vvec;
      uint4* kd = reinterpret_cast<uint4*>(L.kpool) + dst_row * kvec;
      uint4* vd = reinterpret_cast<uint4*>(L.vpool) + dst_row * vvec;
      const int nk = rows * kvec, nvv = d.v_shares_k ? 0 : rows * vvec;
      for (int base = 0; base < vpi; base += 32 * kFetchUnroll) {
        uint4 val[kFetchUnroll];
#pragma unroll
        for (int k = 0; k < kFetchUnroll; ++k) {
          const int w = base + k * 32 + lane;
          if (w < vk ? w < nk : w - vk < nvv) val[k] = w < vk ? ks[w] : vs[w - vk];
        }
#pragma unroll
        for (int k = 0; k < kFetchUnroll; ++k) {
          const int w = base + k * 32 + lane;
          if (w < vk ? w < nk : w - vk < nvv) {
            if (w < vk) kd[w] = val[k]; else vd[w - vk] = val[k];
          }
        }
      }
    }
  }
  for (int batch = gwarp; !SINGLE && batch < n_batches; batch += nwarps) {
    const int i0 = batch * ipb, ni = min(ipb, total - i0);
    // lane k < ni locates item i0 + k: unit by binary search over s_off, then its block and slot
    int my_u = 0, my_rows = 0;
    size_t my_src = 0, my_dst = 0;
    if (lane < ni) {
      int item = i0 + lane;
      int lo = 0, hi = d.U;                               // s_off[lo] <= item < s_off[hi]
      while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (s_off[mid] <= item) lo = mid; else hi = mid;
      }
      my_u = lo;
      const int j = item - s_off[lo];
      const int b = L.fetch_blk[(size_t)lo * d.C + j], s = L.fetch_slot[(size_t)lo * d.C + j];
      const int len = ctx_len[lo / d.Hkv];
      my_rows = max(0, min(d.bs, len - b * d.bs));
      my_src = (size_t)lo * d.max_ctx + (size_t)b * d.bs;   // first host row of the block
      my_dst = ((size_t)lo * d.C + s) * d.bs;               // first slot row
    }
    const int nv = ni * vpi;
    for (int base = 0; base < nv; base += 32 * kFetchUnroll) {
      uint4 val[kFetchUnroll];
      const uint4* src[kFetchUnroll];
      uint4* dst[kFetchUnroll];
#pragma unroll
      for (int k = 0; k < kFetchUnroll; ++k) {
        const int f = base + k * 32 + lane;
        const int it = f / vpi, w = f - (f / vpi) * vpi;
        const int rows = __shfl_sync(0xffffffffu, my_rows, it < ni ? it : 0);
        const size_t sr = __shfl_sync(0xffffffffu, my_src, it < ni ? it : 0);
        const size_t dr = __shfl_sync(0xffffffffu, my_dst, it < ni ? it : 0);
        src[k] = nullptr;
        dst[k] = nullptr;
        if (f < nv) {
          if (w < vk) {
            if (w < rows * kvec) {
              src[k] = reinterpret_cast<const uint4*>(L.host_k) + sr * kvec + w;
              dst[k] = reinterpret_cast<uint4*>(L.kpool) + dr * kvec + w;
            }
          } else {
            const int w2 = w - vk;
            if (w2 < rows * vvec) {
              src[k] = reinterpret_cast<const uint4*>(L.host_v) + sr * vvec + w2;
              dst[k] = reinterpret_cast<uint4*>(L.vpool) + dr * vvec + w2;
            }
          }
        }
        if (src[k]) val[k] = *src[k];
      }
#pragma unroll
      for (int k = 0; k < kFetchUnroll; ++k)
        if (dst[k]) *dst[k] = val[k];
    }
  }
  // lookahead: commit the selections the update staged (this kernel runs after the layer's
  // attention over the previous pending selection; done after the copies, which do not depend on
  // it, so that the host reads start at once); unit u is handled by CTA u % grid
  if (d.lookahead) {
    for (int u = blockIdx.x; u < d.U; u += gridDim.x) {
      const int commit = L.next_commit[u];
      __syncthreads();   // every thread has read the flag before thread 0 clears it
      if (!commit) continue;
      const int n = L.next_n[u];
      for (int i = tid; i < n; i += blockDim.x) {
        L.pend_sel[(size_t)u * d.Kb + i] = L.next_sel[(size_t)u * d.Kb + i];
        L.pend_slot[(size_t)u * d.Kb + i] = L.next_slot[(size_t)u * d.Kb + i];
      }
      if (tid == 0) {
        L.pend_n[u] = n;
        L.next_commit[u] = 0;
      }
    }
  }
}

}  // namespace

cudaError_t launch_cache_update(const Dims& d, const Layer& L, const int* sel, const int* nsel, const int* ctx_len,
                                int* slot_of_sel, const float* scores, kvs_stats* stats, cudaStream_t s) {
  size_t smem = update_smem_bytes(d);
  {   // always, not only above 48 KB: with the kernel's static shared memory the total may pass it
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(cache_update_kernel), (int)smem);
    if (e != cudaSuccess) return e;
  }
  launch_pdl(cache_update_kernel, dim3(d.U), dim3(kCacheThreads), smem, s, d, L, sel, nsel, ctx_len, slot_of_sel, scores,
             stats);
  return cudaGetLastError();
}

int select_update_fusable(const Dims& d) { return d.nb_max <= kTopkSmemKeys; }

cudaError_t launch_select_update(const Dims& d, const Layer& L, const float* scores, const int* ctx_len, int* sel,
                                 int* nsel, int* slot_of_sel, kvs_stats* stats, cudaStream_t s, int threads) {
  const size_t smem = select_update_smem_bytes(d);
  {   // always, not only above 48 KB: with the kernel's static shared memory the total may pass it
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(select_update_kernel), (int)smem);
    if (e != cudaSuccess) return e;
  }
  launch_pdl(select_update_kernel, dim3(d.U), dim3(threads), smem, s, d, L, scores, ctx_len, sel, nsel,
             slot_of_sel, stats);
  return cudaGetLastError();
}

cudaError_t launch_prefetch(const Dims& d, const Layer& L, const int* hint, const int* hint_n, const int* ctx_len,
                            kvs_stats* stats, cudaStream_t s) {
  size_t smem = cache_smem_bytes(d);
  {   // always, not only above 48 KB: with the kernel's static shared memory the total may pass it
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(prefetch_kernel), (int)smem);
    if (e != cudaSuccess) return e;
  }
  launch_pdl(prefetch_kernel, dim3(d.U), dim3(kCacheThreads), smem, s, d, L, hint, hint_n, ctx_len, stats);
  return cudaGetLastError();
}

SnapshotPlan snapshot_plan(const Dims& d) {
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  SnapshotPlan p;
  const size_t U = d.U;
  p.b2s = al(U * d.nb_max * 4);
  p.s2b = al(U * d.C * 4);
  p.stamp = al(U * d.C * 4);
  p.clock = al(U * 4);
  p.pend_sel = al(U * d.Kb * 4);
  p.pend_slot = al(U * d.Kb * 4);
  p.pend_n = al(U * 4);
  p.total = p.b2s + p.s2b + p.stamp + p.clock + p.pend_sel + p.pend_slot + p.pend_n;
  return p;
}

cudaError_t launch_restore(const Dims& d, const Layer& L, const unsigned char* snap, cudaStream_t s) {
  launch_pdl(restore_kernel, dim3(d.U), dim3(kRestoreThreads), 0, s, d, L, snap, snapshot_plan(d));
  return cudaGetLastError();
}

cudaError_t launch_fetch(const Dims& d, const Layer& L, const int* ctx_len, cudaStream_t s) {
  if (d.U > kFetchMaxUnits) return cudaErrorInvalidValue;
  if (fetch_items_per_batch(d) == 1)
    launch_pdl(fetch_kernel<true>, dim3(device_sm_count()), dim3(kFetchThreads), 0, s, d, L, ctx_len);
  else
    launch_pdl(fetch_kernel<false>, dim3(device_sm_count()), dim3(kFetchThreads), 0, s, d, L, ctx_len);
  return cudaGetLastError();
}

}  // namespace kvs
