// GPU working-set cache of each (request, layer, kv-head) unit: hit detection, the delta of
// missing blocks, least-recently-used victims under the capacity cap, slot assignment and
// stamps (one CTA per unit, so the state of a unit has a single writer), the cross-layer
// prefetch, and the zero-copy host -> slot fetch of the blocks each of them maps.
//
// Stamps are assigned, never incremented: every block of a selection gets 2*clock, a prefetched
// block 2*clock + 1, so the (stamp, slot) order is deterministic.
#include "kvs_block.cuh"
#include "kvs_common.cuh"
#include "kvs_ptx.cuh"
#include "kvs_select.cuh"

#include <algorithm>

namespace kvs {

namespace {

constexpr int kCacheThreads = 512;

struct CacheSmem {
  uint8_t* flags;     // [C]  bit 0: holds a selected (or hint) block, bit 1: pinned
  uint32_t* lt_key;   // [MV] victims strictly below the threshold key (slot order)
  int* lt_slot;       // [MV]
  int* vict;          // [MV] victim slots in LRU order
  int* list_blk;      // [Kb] misses (update) or non-resident hint blocks (prefetch), ascending
  int* list_pos;      // [Kb] position of each miss in the selection
  int* sos;           // [Kb] slot of each selected block
  int* s2b;           // [C]  the unit's slot -> block map, read once (update)
  unsigned* st;       // [C]  the unit's stamps, read once (update)
};

__host__ __device__ inline int max_victims(const Dims& d) { return d.Kb > d.max_prefetch ? d.Kb : d.max_prefetch; }

__host__ __device__ inline size_t cache_smem_bytes(const Dims& d) {
  size_t mv = (size_t)max_victims(d);
  return ((size_t)d.C + 15) / 16 * 16 + mv * 12 + (size_t)d.Kb * 12 + (size_t)d.C * 8;
}

__device__ CacheSmem carve(unsigned char* base, const Dims& d) {
  CacheSmem s;
  size_t mv = (size_t)max_victims(d);
  s.flags = base;
  base += ((size_t)d.C + 15) / 16 * 16;
  s.lt_key = reinterpret_cast<uint32_t*>(base); base += mv * 4;
  s.lt_slot = reinterpret_cast<int*>(base); base += mv * 4;
  s.vict = reinterpret_cast<int*>(base); base += mv * 4;
  s.list_blk = reinterpret_cast<int*>(base); base += (size_t)d.Kb * 4;
  s.list_pos = reinterpret_cast<int*>(base); base += (size_t)d.Kb * 4;
  s.sos = reinterpret_cast<int*>(base); base += (size_t)d.Kb * 4;
  s.s2b = reinterpret_cast<int*>(base); base += (size_t)d.C * 4;
  s.st = reinterpret_cast<unsigned*>(base);
  return s;
}

// The m eligible slots with the smallest (key, slot), in that order, into vict[0 .. m).
// Requires m <= number of eligible slots.
template <class Elig, class Key>
__device__ void select_victims(int C, int m, Elig elig, Key key, int* hist, int* ws, int* pick, CacheSmem& sm) {
  const int tid = threadIdx.x, NT = blockDim.x;
  if (m <= 0) return;
  uint32_t prefix = 0, mask = 0;
  int remaining = m;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += NT) hist[i] = 0;
    __syncthreads();
    for (int s = tid; s < C; s += NT) {
      if (!elig(s)) continue;
      uint32_t k = key(s);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid < 32) radix_pick_digit(hist, remaining, false, pick);
    __syncthreads();
    prefix |= (uint32_t)pick[0] << shift;
    mask |= 255u << shift;
    remaining -= pick[1];
    __syncthreads();
  }
  const uint32_t T = prefix;
  const int need_eq = remaining, n_lt = m - remaining;
  const int per = (C + NT - 1) / NT;
  const int s0 = min(C, tid * per), s1 = min(C, s0 + per);
  int my_lt = 0, my_eq = 0;
  for (int s = s0; s < s1; ++s) {
    if (!elig(s)) continue;
    uint32_t k = key(s);
    my_lt += k < T;
    my_eq += k == T;
  }
  int tot;
  int lt_pos = block_excl_sum(my_lt, ws, &tot);
  int eq_pos = block_excl_sum(my_eq, ws, &tot);
  for (int s = s0; s < s1; ++s) {
    if (!elig(s)) continue;
    uint32_t k = key(s);
    if (k < T) { sm.lt_key[lt_pos] = k; sm.lt_slot[lt_pos] = s; ++lt_pos; }
    else if (k == T) { if (eq_pos < need_eq) sm.vict[n_lt + eq_pos] = s; ++eq_pos; }
  }
  __syncthreads();
  // entries below T are in slot order: rank = #smaller keys + #equal keys earlier in slot order
  for (int i = tid; i < n_lt; i += NT) {
    uint32_t k = sm.lt_key[i];
    int rank = 0;
    for (int j = 0; j < n_lt; ++j) {
      uint32_t kj = sm.lt_key[j];
      rank += (kj < k) || (kj == k && j < i);
    }
    sm.vict[rank] = sm.lt_slot[i];
  }
  __syncthreads();
}

__device__ __forceinline__ unsigned long long fetch_rows(const Dims& d, int len, int b) {
  return (unsigned long long)min(d.bs, len - b * d.bs);
}

struct UpdateShared {
  int hist[256];
  int ws[33];
  int pick[2];
  int bad;
  unsigned long long cnt[4];  // hits, prefetch hits, evictions, bytes
};

// The update stages the unit's block -> slot map in shared memory when it is this small.
__host__ __device__ inline bool update_stages_b2s(const Dims& d) { return d.nb_max <= 16384; }
// Caches of up to this many slots take their victims by counting ranks in one pass.
constexpr int kRankVictimsMaxC = 1024;

// Shared memory of the update: the CacheSmem arrays, then the staged selection and pending
// slots [Kb] each, the victims' (key, slot) words [C], and the staged block -> slot map.
__host__ __device__ inline size_t update_extra_offset(const Dims& d) { return (cache_smem_bytes(d) + 15) / 16 * 16; }
__host__ __device__ inline size_t update_smem_bytes(const Dims& d) {
  return update_extra_offset(d) + (size_t)d.Kb * 8 + (size_t)d.C * 8 + (update_stages_b2s(d) ? (size_t)d.nb_max * 4 : 0);
}

// The cache update of unit u (every thread of the CTA calls it).  Every input that does not depend
// on another is read in one round of loads (the selection, the slot map and stamps, the pending
// slots, the block -> slot map when it is staged); sel and nsel may have been written earlier in
// the same kernel by this CTA (the fused top-K + update), so they are read through plain loads.
__device__ void update_unit(const Dims& d, const Layer& L, int u, const int* sel, const int* nsel,
                            const int* __restrict__ ctx_len, int* __restrict__ slot_of_sel,
                            const float* __restrict__ imp, kvs_stats* stats, unsigned char* smraw, UpdateShared& sh) {
  int* hist = sh.hist;
  int* ws = sh.ws;
  int* pick = sh.pick;
  int& s_bad = sh.bad;
  unsigned long long* s_cnt = sh.cnt;
  CacheSmem sm = carve(smraw, d);
  int* su_s = reinterpret_cast<int*>(smraw + update_extra_offset(d));   // [Kb] the selection
  int* ps_s = su_s + d.Kb;                                             // [Kb] the pending slots
  unsigned long long* ck = reinterpret_cast<unsigned long long*>(ps_s + d.Kb);   // [C] victim (key, slot)
  int* b2s_s = update_stages_b2s(d) ? reinterpret_cast<int*>(ck + d.C) : nullptr;   // [nb_max]
  const int r = u / d.Hkv;
  const int tid = threadIdx.x, NT = blockDim.x;
  int* b2s = L.block2slot + (size_t)u * d.nb_max;
  int* s2b = L.slot2block + (size_t)u * d.C;
  unsigned* st = L.stamp + (size_t)u * d.C;
  const int len = ctx_len[r];
  const int n = nsel[u];
  const int pn = d.lookahead ? L.pend_n[u] : -1;
  const unsigned now = 2u * (L.clock[u] + 1u);   // written back only once the update is accepted
  if (tid == 0) s_bad = 0;
  if (tid < 4) s_cnt[tid] = 0;
  for (int s = tid; s < d.C; s += NT) {
    sm.flags[s] = 0;
    sm.s2b[s] = s2b[s];
    sm.st[s] = st[s];
  }
  for (int i = tid; i < d.Kb; i += NT) {
    su_s[i] = sel[(size_t)u * d.Kb + i];
    ps_s[i] = d.lookahead ? L.pend_slot[(size_t)u * d.Kb + i] : -1;
  }
  if (b2s_s)
    for (int b = tid; b < d.nb_max; b += NT) b2s_s[b] = b2s[b];
  __syncthreads();
  const int nb = n_blocks_of(len, d.bs);
  if (len < 0 || len > d.max_ctx || n < 0 || n > d.Kb) {
    if (tid == 0) {
      set_error(L.err, KVS_ERR_BAD_INDEX);
      L.n_fetch[u] = 0;
      L.next_commit[u] = 0;
    }
    return;
  }
  auto slot_of = [&](int b) { return b2s_s ? b2s_s[b] : b2s[b]; };

  // hits and misses, misses compacted in selection (ascending block) order
  const int per = (n + NT - 1) / NT;
  const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
  int my_miss = 0;
  unsigned long long my_pfh = 0;
  for (int i = i0; i < i1; ++i) {
    int b = su_s[i];
    // a selection is strictly ascending (top-K output order); anything else is refused
    if (b < 0 || b >= nb || (i > 0 && su_s[i - 1] >= b)) { s_bad = 1; continue; }
    int s = slot_of(b);
    if (s >= d.C) { s_bad = 1; continue; }
    if (s >= 0) {
      sm.flags[s] = 1;
      sm.sos[i] = s;
      my_pfh += sm.st[s] == now - 1u;
    } else {
      ++my_miss;
    }
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      set_error(L.err, KVS_ERR_BAD_INDEX);
      L.n_fetch[u] = 0;
      L.next_commit[u] = 0;
    }
    return;
  }
  int m;
  int mpos = block_excl_sum(my_miss, ws, &m);
  for (int i = i0; i < i1; ++i) {
    int b = su_s[i];
    if (slot_of(b) < 0) { sm.list_blk[mpos] = b; sm.list_pos[mpos] = i; ++mpos; }
  }
  const bool pinned = d.lookahead && pn >= 0;
  if (pinned) {
    for (int i = tid; i < pn && i < d.Kb; i += NT) {
      int s = ps_s[i];
      if (s >= 0 && s < d.C) sm.flags[s] |= 2;
    }
  }
  if (my_pfh) atomicAdd(&s_cnt[1], my_pfh);
  __syncthreads();

  // eligible slots with and without the pins, in one prefix sum (both counts are below 2^16)
  int my_el = 0, my_el_nopin = 0;   // C <= 8192
  for (int s = tid; s < d.C; s += NT) {
    my_el += sm.flags[s] == 0;
    my_el_nopin += (sm.flags[s] & 1) == 0;
  }
  int both;
  block_excl_sum(my_el | (my_el_nopin << 16), ws, &both);
  int n_el = both & 0xffff;
  const int n_el_nopin = both >> 16;
  bool fallback = false;
  if (n_el < m && pinned) { fallback = true; n_el = n_el_nopin; }
  if (n_el < m) {
    if (tid == 0) {
      set_error(L.err, KVS_ERR_CAPACITY);
      L.n_fetch[u] = 0;
      L.next_commit[u] = 0;
    }
    return;
  }
  // accepted: a refused update (bad index, capacity) leaves the unit's state as it was
  if (tid == 0) L.clock[u] = now / 2u;
  const uint8_t emask = fallback ? 1 : 3;
  // victim keys, smallest first: empty slots 0; LRU: the stamp (>= 2); importance: 1 + the
  // orderable key of the held block's score (NaN lowest), so the least important go first
  const float* imp_u = imp ? imp + (size_t)u * d.nb_max : nullptr;
  auto elig = [&](int s) { return (sm.flags[s] & emask) == 0; };
  auto vkey = [&](int s) {
    const int b = sm.s2b[s];
    if (b < 0) return 0u;
    return imp_u ? score_key(imp_u[b]) + 1u : sm.st[s];
  };
  if (d.C <= kRankVictimsMaxC) {
    // the m smallest (key, slot) among the eligible slots by rank counting: one word per slot,
    // all-ones for ineligible ones (never below an eligible word)
    for (int s = tid; s < d.C; s += NT) ck[s] = elig(s) ? ((unsigned long long)vkey(s) << 32) | (unsigned)s : ~0ull;
    __syncthreads();
    for (int s = tid; s < d.C; s += NT) {
      const unsigned long long mine = ck[s];
      if (mine == ~0ull) continue;
      int rank = 0;
      for (int t = 0; t < d.C; ++t) rank += ck[t] < mine;
      if (rank < m) sm.vict[rank] = s;
    }
    __syncthreads();
  } else {
    select_victims(d.C, m, elig, vkey, hist, ws, pick, sm);
  }

  unsigned long long my_ev = 0, my_bytes = 0;
  for (int j = tid; j < m; j += NT) {
    int b = sm.list_blk[j], s = sm.vict[j];
    int old = sm.s2b[s];
    if (old >= 0 && old < d.nb_max) { b2s[old] = -1; ++my_ev; }
    s2b[s] = b;
    b2s[b] = s;
    sm.sos[sm.list_pos[j]] = s;
    L.fetch_blk[(size_t)u * d.C + j] = b;
    L.fetch_slot[(size_t)u * d.C + j] = s;
    my_bytes += fetch_rows(d, len, b) * (unsigned long long)d.row_bytes;
  }
  if (my_ev) atomicAdd(&s_cnt[2], my_ev);
  if (my_bytes) atomicAdd(&s_cnt[3], my_bytes);
  __syncthreads();
  for (int i = tid; i < n; i += NT) {
    int s = sm.sos[i];
    st[s] = now;
    slot_of_sel[(size_t)u * d.Kb + i] = s;
    if (d.lookahead) {   // staged; the fetch that follows commits it to pend_*
      L.next_sel[(size_t)u * d.Kb + i] = su_s[i];
      L.next_slot[(size_t)u * d.Kb + i] = s;
    }
  }
  if (tid == 0) {
    L.n_fetch[u] = m;
    if (d.lookahead) {
      L.next_n[u] = n;
      L.next_commit[u] = 1;
    }
    if (stats) {
      kvs_stats* sl = stats + L.layer;
      atomicAdd(&sl->hits, (unsigned long long)(n - m));
      atomicAdd(&sl->misses, (unsigned long long)m);
      atomicAdd(&sl->prefetch_hits, s_cnt[1]);
      atomicAdd(&sl->evictions, s_cnt[2]);
      atomicAdd(&sl->bytes_fetched, s_cnt[3]);
      if (fallback) atomicAdd(&sl->pin_fallbacks, 1ull);
    }
  }
}

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
// blocks): the selection goes to sel / nsel as from the top-K kernel, and the update reads it
// back after a barrier, with no kernel boundary between the two.
__global__ void __launch_bounds__(kCacheThreads) select_update_kernel(Dims d, Layer L, const float* __restrict__ scores,
                                                                      const int* __restrict__ ctx_len, int* sel,
                                                                      int* nsel, int* __restrict__ slot_of_sel,
                                                                      kvs_stats* stats) {
  kvs_pdl_entry();
  extern __shared__ __align__(16) unsigned char smraw[];
  __shared__ TopkShared tsh;
  __shared__ UpdateShared ush;
  const int u = blockIdx.x;
  topk_unit_smem(d, scores, ctx_len[u / d.Hkv], u, sel, nsel, L.err, reinterpret_cast<uint32_t*>(smraw), tsh);
  __syncthreads();   // the selection (global) and the key buffer (shared, reused below) are done
  update_unit(d, L, u, sel, nsel, ctx_len, slot_of_sel, d.evict_importance ? scores : nullptr, stats, smraw, ush);
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
  if (smem > 48 * 1024) {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(cache_update_kernel), (int)smem);
    if (e != cudaSuccess) return e;
  }
  launch_pdl(cache_update_kernel, dim3(d.U), dim3(kCacheThreads), smem, s, d, L, sel, nsel, ctx_len, slot_of_sel, scores,
             stats);
  return cudaGetLastError();
}

int select_update_fusable(const Dims& d) { return d.nb_max <= kTopkSmemKeys; }

cudaError_t launch_select_update(const Dims& d, const Layer& L, const float* scores, const int* ctx_len, int* sel,
                                 int* nsel, int* slot_of_sel, kvs_stats* stats, cudaStream_t s) {
  const size_t smem = std::max(update_smem_bytes(d), (size_t)d.nb_max * sizeof(uint32_t));
  if (smem > 48 * 1024) {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(select_update_kernel), (int)smem);
    if (e != cudaSuccess) return e;
  }
  launch_pdl(select_update_kernel, dim3(d.U), dim3(kCacheThreads), smem, s, d, L, scores, ctx_len, sel, nsel,
             slot_of_sel, stats);
  return cudaGetLastError();
}

cudaError_t launch_prefetch(const Dims& d, const Layer& L, const int* hint, const int* hint_n, const int* ctx_len,
                            kvs_stats* stats, cudaStream_t s) {
  size_t smem = cache_smem_bytes(d);
  if (smem > 48 * 1024) {
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
