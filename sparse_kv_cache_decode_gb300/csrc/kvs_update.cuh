// The cache update of one (request, layer, kv-head) unit by one CTA: hit detection, the delta of
// missing blocks, victims under the capacity cap (least recently used, or least important), slot
// assignment and stamps.  Shared by the update kernels and the fused layer kernel.
//
// Stamps are assigned, never incremented: every block of a selection gets 2*clock, a prefetched
// block 2*clock + 1, so the (stamp, slot) order is deterministic.
#pragma once
#include "kvs_block.cuh"
#include "kvs_common.cuh"
#include "kvs_ptx.cuh"
#include "kvs_select.cuh"

namespace kvs {

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

__device__ inline CacheSmem carve(unsigned char* base, const Dims& d) {
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
__device__ inline void select_victims(int C, int m, Elig elig, Key key, int* hist, int* ws, int* pick, CacheSmem& sm) {
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
  int n_ck;                   // eligible slots gathered for the victim ranking
  unsigned long long cnt[4];  // hits, prefetch hits, evictions, bytes
};

// The update stages the unit's block -> slot map in shared memory when it is this small.
__host__ __device__ inline bool update_stages_b2s(const Dims& d) { return d.nb_max <= 16384; }
// Caches of up to this many slots take their victims by counting ranks in one pass.
constexpr int kRankVictimsMaxC = 1024;

// Shared memory of the update: the CacheSmem arrays, then the staged selection and pending
// slots [Kb] each, the victims' (key, slot) words [C], and the staged block -> slot map.
__host__ __device__ inline size_t update_extra_offset(const Dims& d) { return (cache_smem_bytes(d) + 15) / 16 * 16; }
__host__ __device__ inline size_t update_missf_offset(const Dims& d) {
  return update_extra_offset(d) + (size_t)d.Kb * 8 + (size_t)d.C * 8 + (update_stages_b2s(d) ? (size_t)d.nb_max * 4 : 0);
}
__host__ __device__ inline size_t update_smem_bytes(const Dims& d) {
  return update_missf_offset(d) + ((size_t)d.Kb + 15) / 16 * 16;   // + the per-position miss flags
}

// Inputs of the update that do not depend on the selection (per-thread copies of the scalars).
struct UpdateIn {
  int len, n, pn;
  unsigned clk;
};

// The staged selection of the update in its shared memory: su_s[0 .. n).
__device__ __forceinline__ int* update_sel_buffer(const Dims& d, unsigned char* smraw) {
  return reinterpret_cast<int*>(smraw + update_extra_offset(d));
}

// Phase 1 of the cache update of unit u: issues the reads of every input that does not depend on
// the selection (the slot map and stamps, the pending slots, the block -> slot map when it is
// staged) into shared memory, through L2, and returns the scalars (n is left 0).  It does not wait:
// the caller fills the selection, waits for its copies (cp_async_wait_all) and synchronises the CTA
// before update_run.  Every thread of the CTA calls it.
__device__ inline UpdateIn update_stage(const Dims& d, const Layer& L, int u, const int* __restrict__ ctx_len,
                                        unsigned char* smraw, UpdateShared& sh) {
  CacheSmem sm = carve(smraw, d);
  int* ps_s = update_sel_buffer(d, smraw) + d.Kb;
  unsigned long long* ck = reinterpret_cast<unsigned long long*>(ps_s + d.Kb);
  int* b2s_s = update_stages_b2s(d) ? reinterpret_cast<int*>(ck + d.C) : nullptr;
  const int tid = threadIdx.x, NT = blockDim.x;
  UpdateIn in;
  in.len = ctx_len[u / d.Hkv];
  in.n = 0;
  in.pn = d.lookahead ? __ldcg(L.pend_n + u) : -1;
  in.clk = __ldcg(L.clock + u);
  if (tid == 0) sh.bad = 0;
  if (tid < 4) sh.cnt[tid] = 0;
  for (int s = tid; s < d.C; s += NT) sm.flags[s] = 0;
  stage_words(sm.s2b, L.slot2block + (size_t)u * d.C, d.C);
  stage_words(sm.st, L.stamp + (size_t)u * d.C, d.C);
  if (d.lookahead)
    stage_words(ps_s, L.pend_slot + (size_t)u * d.Kb, d.Kb);
  else
    for (int i = tid; i < d.Kb; i += NT) ps_s[i] = -1;
  if (b2s_s) stage_words(b2s_s, L.block2slot + (size_t)u * d.nb_max, d.nb_max);
  return in;
}

// Phase 2: the update itself, from shared memory (after update_stage, the selection in
// update_sel_buffer, the copies waited for and a CTA barrier); in.n is the selection's count.
// The scores (importance eviction) are read through L2, as other CTAs of the kernel may have
// written them.
__device__ inline void update_run(const Dims& d, const Layer& L, int u, const UpdateIn& in,
                                  int* __restrict__ slot_of_sel, const float* imp, kvs_stats* stats,
                                  unsigned char* smraw, UpdateShared& sh) {
  int* hist = sh.hist;
  int* ws = sh.ws;
  int* pick = sh.pick;
  int& s_bad = sh.bad;
  unsigned long long* s_cnt = sh.cnt;
  CacheSmem sm = carve(smraw, d);
  int* su_s = update_sel_buffer(d, smraw);                             // [Kb] the selection
  int* ps_s = su_s + d.Kb;                                             // [Kb] the pending slots
  unsigned long long* ck = reinterpret_cast<unsigned long long*>(ps_s + d.Kb);   // [C] victim (key, slot)
  int* b2s_s = update_stages_b2s(d) ? reinterpret_cast<int*>(ck + d.C) : nullptr;   // [nb_max]
  uint8_t* mf_s = smraw + update_missf_offset(d);                      // [Kb] position i missed
  const int tid = threadIdx.x, NT = blockDim.x;
  int* b2s = L.block2slot + (size_t)u * d.nb_max;
  int* s2b = L.slot2block + (size_t)u * d.C;
  unsigned* st = L.stamp + (size_t)u * d.C;
  const int len = in.len, n = in.n, pn = in.pn;
  const unsigned now = 2u * (in.clk + 1u);   // written back only once the update is accepted
  const int nb = n_blocks_of(len, d.bs);
  if (len < 0 || len > d.max_ctx || n < 0 || n > d.Kb) {
    if (tid == 0) {
      set_error(L.err, KVS_ERR_BAD_INDEX);
      L.n_fetch[u] = 0;
      L.next_commit[u] = 0;
    }
    return;
  }
  auto slot_of = [&](int b) { return b2s_s ? b2s_s[b] : __ldcg(b2s + b); };

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
      mf_s[i] = 0;
      sm.sos[i] = s;
      my_pfh += sm.st[s] == now - 1u;
    } else {
      ++my_miss;
      mf_s[i] = 1;
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
    return imp_u ? score_key(__ldcg(imp_u + b)) + 1u : sm.st[s];
  };
  if (d.C <= kRankVictimsMaxC) {
    // the m smallest (key, slot) among the eligible slots by rank counting: the eligible slots'
    // (key, slot) words are gathered first (in any order: a rank depends only on the values), then
    // each is ranked against the others
    if (tid == 0) sh.n_ck = 0;
    __syncthreads();
    const int lane = tid & 31;
    for (int s0 = tid - lane; s0 < d.C; s0 += NT) {   // warp-uniform trip count
      const int s = s0 + lane;
      const bool e = s < d.C && elig(s);
      const unsigned em = __ballot_sync(0xffffffffu, e);
      int base = 0;
      if (lane == 0 && em) base = atomicAdd(&sh.n_ck, __popc(em));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (e) ck[base + __popc(em & ((1u << lane) - 1u))] = ((unsigned long long)vkey(s) << 32) | (unsigned)s;
    }
    __syncthreads();
    const int ne = sh.n_ck;
    for (int i = tid; i < ne; i += NT) {
      const unsigned long long mine = ck[i];
      int rank = 0;
      for (int t = 0; t < ne; ++t) rank += ck[t] < mine;
      if (rank < m) sm.vict[rank] = (int)(mine & 0xffffffffu);
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
    L.miss_flag[(size_t)u * d.Kb + i] = mf_s[i];
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

// Top-K + update of one unit in one CTA: the update's shared memory, then the unit's score row
// (nb_max words, turned into keys in place) from a 16-byte aligned offset, then the top-K's
// threshold-guess scratch.
__host__ __device__ inline size_t select_keys_offset(const Dims& d) { return (update_smem_bytes(d) + 15) / 16 * 16; }
__host__ __device__ inline size_t select_scratch_offset(const Dims& d) {
  return (select_keys_offset(d) + (size_t)d.nb_max * 4 + 15) / 16 * 16;
}
__host__ __device__ inline size_t select_update_smem_bytes(const Dims& d) {
  return select_scratch_offset(d) + (size_t)kTopkFastScratch * 4;
}

// The cache update of unit u with the selection read from sel / nsel (every thread of the CTA
// calls it; sel and nsel may have been written earlier in the same kernel by this CTA, so they
// are read through plain loads).
__device__ inline void update_unit(const Dims& d, const Layer& L, int u, const int* sel, const int* nsel,
                                   const int* __restrict__ ctx_len, int* __restrict__ slot_of_sel, const float* imp,
                                   kvs_stats* stats, unsigned char* smraw, UpdateShared& sh) {
  UpdateIn in = update_stage(d, L, u, ctx_len, smraw, sh);
  in.n = nsel[u];
  int* su_s = update_sel_buffer(d, smraw);
  for (int i = threadIdx.x; i < d.Kb; i += blockDim.x) su_s[i] = sel[(size_t)u * d.Kb + i];
  cp_async_wait_all();
  __syncthreads();
  update_run(d, L, u, in, slot_of_sel, imp, stats, smraw, sh);
}

}  // namespace kvs
