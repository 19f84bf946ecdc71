// libkvs host side: configuration checks, workspace carving and the C-ABI entry points.
#include <math.h>

#include <algorithm>
#include <stdio.h>
#include <string.h>

#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include <cudaTypedefs.h>

#include "kvs_common.cuh"

using namespace kvs;

struct kvs_ctx {
  kvs_config cfg;
  Dims d;
  unsigned char* ws;
  size_t ws_bytes;
  std::vector<Layer> layers;
  unsigned* err;
  const __nv_bfloat16* host_k_dev;  // whole host history, device-mapped
  const __nv_bfloat16* host_v_dev;
  std::vector<int> booted;          // lookahead: layer has a pending selection
  std::vector<cudaEvent_t> fetch_done;
  std::vector<int> fetch_pending;
  // cross-layer prefetch ordering: a layer's selection is ready (after its top-K), and the
  // prefetch into a layer is done (before that layer's update); flags cleared by kvs_join
  std::vector<cudaEvent_t> sel_ready, pf_done;
  std::vector<int> sel_pending, pf_pending;
  std::vector<CUtensorMap> tmaps;   // per layer: K pool, V pool (TMA attention path)
  // two-phase top-K candidates (long contexts), one copy per layer parity (like the block scores)
  kvs::TopkScratch tk[2] = {};
  // overlapped lookahead steps: two selection-chain streams (even and odd layers, so that a layer's
  // chain need not wait for the chain of the layer below), and per layer the events that order
  // them (start after the layer below's attention; update done; attention done)
  cudaStream_t sel_stream[2] = {nullptr, nullptr};
  std::vector<cudaEvent_t> layer_start, upd_done, attn_done;
  // diagnostics
  unsigned long long launches = 0;
  struct Timer {
    int count = 0;
    std::vector<cudaEvent_t> start, stop;
  };
  Timer timers[KVS_K_INDEX + 1];
};

namespace {

constexpr size_t kAlign = 256;

// the appended token's rows are read and written as 16-byte vectors
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool fill_dims(const kvs_config* c, Dims* d) {
  if (!c) return false;
  if (c->n_req < 1 || c->n_layer < 1 || c->n_q_head < 1 || c->n_kv_head < 1) return false;
  if (c->n_q_head % c->n_kv_head) return false;
  if (c->n_req > 4096 || c->n_layer > 1024 || c->n_kv_head > 1024) return false;
  if ((long long)c->n_req * c->n_kv_head > 1024) return false;   // units per layer
  if (c->d_k < 8 || c->d_k % 8 || c->d_v < 8 || c->d_v % 8) return false;
  if (c->v_shares_k != 0 && c->v_shares_k != 1) return false;
  if (c->v_shares_k && c->d_v > c->d_k) return false;
  if (c->block_size < 1 || c->max_ctx < 1) return false;
  if (c->budget_blocks < 1 || c->n_sink < 0 || c->n_recent < 0) return false;
  if (c->n_sink + c->n_recent > c->budget_blocks) return false;
  if (c->budget_blocks > 4096) return false;
  if (c->cap_blocks < c->budget_blocks || c->cap_blocks > 8192) return false;
  if (c->max_score_q < 1 || c->max_score_q > 64) return false;
  if (c->lookahead != 0 && c->lookahead != 1) return false;
  if (c->max_prefetch < 0 || c->max_prefetch > c->cap_blocks - c->budget_blocks) return false;
  if (!(c->softmax_scale >= 0.f) || isinf(c->softmax_scale)) return false;
  if (c->evict_policy != KVS_EVICT_LRU && c->evict_policy != KVS_EVICT_IMPORTANCE) return false;
  if (c->score_mode != KVS_SCORE_MEAN && c->score_mode != KVS_SCORE_BOUND) return false;
  if (c->kv_dtype != KVS_KV_BF16 && c->kv_dtype != KVS_KV_FP8_E4M3) return false;
  if (c->kv_dtype == KVS_KV_FP8_E4M3) {
    // E4M3 history: block-mean scoring, separate K and V, rows of whole 16-byte vectors
    if (c->score_mode != KVS_SCORE_MEAN || c->v_shares_k || c->d_k % 16 || c->d_v % 16) return false;
    if (!(c->k_scale >= 0.f) || !(c->v_scale >= 0.f) || isinf(c->k_scale) || isinf(c->v_scale)) return false;
  }
  d->B = c->n_req;
  d->NL = c->n_layer;
  d->Hq = c->n_q_head;
  d->Hkv = c->n_kv_head;
  d->G = c->n_q_head / c->n_kv_head;
  d->dk = c->d_k;
  d->dv = c->d_v;
  d->v_shares_k = c->v_shares_k;
  d->bs = c->block_size;
  d->max_ctx = c->max_ctx;
  d->nb_max = (c->max_ctx + c->block_size - 1) / c->block_size;
  d->Kb = c->budget_blocks;
  d->n_sink = c->n_sink;
  d->n_recent = c->n_recent;
  d->C = c->cap_blocks;
  d->max_nq = c->max_score_q;
  d->lookahead = c->lookahead;
  d->max_prefetch = c->max_prefetch ? c->max_prefetch : c->cap_blocks - c->budget_blocks;
  d->U = c->n_req * c->n_kv_head;
  d->scale = c->softmax_scale > 0.f ? c->softmax_scale : (float)(1.0 / sqrt((double)c->d_k));
  d->timeout_us = c->wait_timeout_us ? c->wait_timeout_us : 2000000u;
  d->fp8 = c->kv_dtype == KVS_KV_FP8_E4M3;
  d->ebytes = d->fp8 ? 1 : 2;
  d->k_scale = d->fp8 && c->k_scale > 0.f ? c->k_scale : 1.f;
  d->v_scale = d->fp8 && c->v_scale > 0.f ? c->v_scale : 1.f;
  d->row_bytes = d->ebytes * (c->d_k + (c->v_shares_k ? 0 : c->d_v));
  d->evict_importance = c->evict_policy == KVS_EVICT_IMPORTANCE;
  d->bound = c->score_mode == KVS_SCORE_BOUND;
  d->didx = d->bound ? 2 * c->d_k : c->d_k;
  return true;
}

// Byte sizes of the per-layer and shared workspace regions.
struct Plan {
  size_t kpool, vpool, b2s, s2b, stamp, clock, pend_sel, pend_slot, pend_n, sel, nsel, sos, fblk, fslot, nfetch;
  size_t next_sel, next_slot, next_n, next_commit, mflag;
  size_t per_layer;
  size_t err, scores, part, ml, done, tk_key, tk_idx, tk_cnt;
  size_t total;
};

Plan plan_of(const Dims& d) {
  Plan p;
  size_t U = d.U;
  p.kpool = align_up(U * d.C * d.bs * (size_t)d.dk * d.ebytes);
  p.vpool = d.v_shares_k ? 0 : align_up(U * d.C * d.bs * (size_t)d.dv * d.ebytes);
  p.b2s = align_up(U * d.nb_max * 4);
  p.s2b = align_up(U * d.C * 4);
  p.stamp = align_up(U * d.C * 4);
  p.clock = align_up(U * 4);
  p.pend_sel = align_up(U * d.Kb * 4);
  p.pend_slot = align_up(U * d.Kb * 4);
  p.pend_n = align_up(U * 4);
  p.sel = align_up(U * d.Kb * 4);
  p.nsel = align_up(U * 4);
  p.sos = align_up(U * d.Kb * 4);
  p.fblk = align_up(U * d.C * 4);
  p.fslot = align_up(U * d.C * 4);
  p.nfetch = align_up(U * 4);
  p.next_sel = align_up(U * d.Kb * 4);
  p.next_slot = align_up(U * d.Kb * 4);
  p.next_n = align_up(U * 4);
  p.next_commit = align_up(U * 4);
  p.mflag = align_up(U * d.Kb);
  p.per_layer = p.kpool + p.vpool + p.b2s + p.s2b + p.stamp + p.clock + p.pend_sel + p.pend_slot + p.pend_n + p.sel +
                p.nsel + p.sos + p.fblk + p.fslot + p.nfetch + p.next_sel + p.next_slot + p.next_n + p.next_commit + p.mflag;
  p.err = align_up(16);
  p.scores = 2 * align_up(U * d.nb_max * 4);   // one copy per layer parity
  size_t parts = kAttnSplitMax;
  if (attention_tma_supported(d)) parts = std::max<size_t>(parts, (size_t)attention_tma_partials(d));
  p.part = align_up(U * parts * d.G * d.dv * 4);
  p.ml = align_up(U * parts * d.G * 2 * 4);
  p.done = align_up(U * 8);   // attention and scoring completion counters, U each
  const size_t P = (size_t)topk_chunks(d);
  p.tk_key = 2 * align_up(U * P * d.Kb * 4);   // one copy per layer parity
  p.tk_idx = 2 * align_up(U * P * d.Kb * 4);
  p.tk_cnt = 2 * align_up(U * P * 4);
  p.total = p.per_layer * d.NL + p.err + p.scores + p.part + p.ml + p.done + p.tk_key + p.tk_idx + p.tk_cnt;
  return p;
}

}  // namespace

namespace kvs {
bool config_to_dims(const kvs_config* c, Dims* d) { return fill_dims(c, d); }

cudaError_t set_max_dynamic_smem(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> set_to;   // (kernel, device) -> bytes allowed
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_pair(kernel, dev);
  auto it = set_to.find(key);
  if (it != set_to.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) set_to[key] = bytes;
  return e;
}

int device_sm_count() {
  static std::mutex mu;
  static std::map<int, int> count;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  std::lock_guard<std::mutex> lock(mu);
  auto it = count.find(dev);
  if (it != count.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 152;
  }
  count[dev] = n;
  return n;
}
}  // namespace kvs

namespace {

inline kvs_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVS_OK : KVS_ERR_CUDA; }

inline bool layer_ok(const kvs_ctx* c, int layer) { return c && layer >= 0 && layer < c->d.NL; }

// Brackets one launcher call with the armed timer's events and counts its kernels.
template <class F>
cudaError_t timed(kvs_ctx* c, int kernel, cudaStream_t s, int n_kernels, F&& launch) {
  kvs_ctx::Timer* t = (kernel > 0 && kernel <= KVS_K_INDEX) ? &c->timers[kernel] : nullptr;
  bool on = t && t->count < (int)t->start.size();
  cudaError_t e = cudaSuccess;
  // inside a stream capture the records must be external to become event-record nodes
  unsigned flags = cudaEventRecordDefault;
  if (on) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(s, &cap);
    if (cap == cudaStreamCaptureStatusActive) flags = cudaEventRecordExternal;
  }
  if (on && e == cudaSuccess) e = cudaEventRecordWithFlags(t->start[t->count], s, flags);
  if (e == cudaSuccess) e = launch();
  if (e == cudaSuccess && on) {
    e = cudaEventRecordWithFlags(t->stop[t->count], s, flags);
    ++t->count;
  }
  if (e == cudaSuccess) c->launches += n_kernels;
  return e;
}

int attn_kernels(const Dims& d) {
  // attention kernel (the TMA and tensor-memory MLA paths merge their partials in-kernel), plus the
  // split combine of the cp.async paths when the selection is split across CTAs
  if (attention_tma_supported(d) || attention_mla_tc_supported(d)) return 1;
  int n_split = 1, bps = 0;
  if (!attention_split(d, &n_split, &bps)) return 1;
  return n_split > 1 ? 2 : 1;
}

inline cudaStream_t S(kvs_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

namespace kvs {
// 2D tensor map over a row-major matrix [rows][inner] of bf16 (elem_bytes 2) or bytes (1), boxes of
// box_inner x box_rows with the 128-byte swizzle (box_inner * elem_bytes must be 128).
bool make_tmap_2d(CUtensorMap* m, void* base, uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows,
                  int elem_bytes) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
      cudaGetLastError();
      return false;
    }
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner * elem_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(m, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base,
                      dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
}  // namespace kvs

namespace {

// The slot pools for the TMA attention kernel's tiles: E4M3 pools as [U*C*bs][128] with 16-row
// boxes (a row is 128 bytes); bf16 pools as lines of 128 bytes, [U*C*bs*d/64][64], with 32-line
// boxes, so that one tensor load brings all 16 rows of a tile.
bool make_pool_map(CUtensorMap* m, void* base, size_t rows, int d, int elem_bytes) {
  if (elem_bytes == 1) return kvs::make_tmap_2d(m, base, (uint64_t)d, (uint64_t)rows, 128, 16, 1);
  return kvs::make_tmap_2d(m, base, 64, (uint64_t)rows * (d / 64), 64, 16 * (d / 64), 2);
}

}  // namespace

extern "C" {

const char* kvs_version(void) { return "kvs 0.1 (sm_103a)"; }

size_t kvs_workspace_bytes(const kvs_config* cfg) {
  Dims d;
  if (!fill_dims(cfg, &d)) return 0;
  return plan_of(d).total;
}

kvs_status kvs_create(const kvs_config* cfg, void* d_workspace, size_t workspace_bytes, kvs_ctx** out) {
  if (!out) return KVS_ERR_INVALID_ARG;
  *out = nullptr;
  Dims d;
  if (!fill_dims(cfg, &d)) return KVS_ERR_INVALID_ARG;
  Plan p = plan_of(d);
  if (!d_workspace || workspace_bytes < p.total || (reinterpret_cast<uintptr_t>(d_workspace) % kAlign))
    return KVS_ERR_INVALID_ARG;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, d_workspace) != cudaSuccess || attr.type != cudaMemoryTypeDevice) {
    cudaGetLastError();
    return KVS_ERR_INVALID_ARG;
  }
  kvs_ctx* c = new (std::nothrow) kvs_ctx();
  if (!c) return KVS_ERR_INVALID_ARG;
  c->cfg = *cfg;
  c->d = d;
  c->ws = static_cast<unsigned char*>(d_workspace);
  c->ws_bytes = workspace_bytes;
  c->host_k_dev = c->host_v_dev = nullptr;
  unsigned char* base = c->ws;
  c->layers.resize(d.NL);
  unsigned char* shared = base + p.per_layer * d.NL;
  c->err = reinterpret_cast<unsigned*>(shared);
  float* scores = reinterpret_cast<float*>(shared + p.err);
  float* part = reinterpret_cast<float*>(shared + p.err + p.scores);
  float* ml = reinterpret_cast<float*>(shared + p.err + p.scores + p.part);
  unsigned* done = reinterpret_cast<unsigned*>(shared + p.err + p.scores + p.part + p.ml);
  unsigned char* tk = shared + p.err + p.scores + p.part + p.ml + p.done;
  for (int par = 0; par < 2; ++par) {
    c->tk[par].key = p.tk_key ? reinterpret_cast<uint32_t*>(tk + par * (p.tk_key / 2)) : nullptr;
    c->tk[par].idx = p.tk_key ? reinterpret_cast<int*>(tk + p.tk_key + par * (p.tk_idx / 2)) : nullptr;
    c->tk[par].cnt = p.tk_key ? reinterpret_cast<int*>(tk + p.tk_key + p.tk_idx + par * (p.tk_cnt / 2)) : nullptr;
  }
  for (int l = 0; l < d.NL; ++l) {
    unsigned char* b = base + p.per_layer * l;
    Layer& L = c->layers[l];
    L.layer = l;
    L.kpool = reinterpret_cast<__nv_bfloat16*>(b); b += p.kpool;
    L.vpool = d.v_shares_k ? nullptr : reinterpret_cast<__nv_bfloat16*>(b); b += p.vpool;
    L.block2slot = reinterpret_cast<int*>(b); b += p.b2s;
    L.slot2block = reinterpret_cast<int*>(b); b += p.s2b;
    L.stamp = reinterpret_cast<unsigned*>(b); b += p.stamp;
    L.clock = reinterpret_cast<unsigned*>(b); b += p.clock;
    L.pend_sel = reinterpret_cast<int*>(b); b += p.pend_sel;
    L.pend_slot = reinterpret_cast<int*>(b); b += p.pend_slot;
    L.pend_n = reinterpret_cast<int*>(b); b += p.pend_n;
    L.sel = reinterpret_cast<int*>(b); b += p.sel;
    L.nsel = reinterpret_cast<int*>(b); b += p.nsel;
    L.slot_of_sel = reinterpret_cast<int*>(b); b += p.sos;
    L.fetch_blk = reinterpret_cast<int*>(b); b += p.fblk;
    L.fetch_slot = reinterpret_cast<int*>(b); b += p.fslot;
    L.n_fetch = reinterpret_cast<int*>(b); b += p.nfetch;
    L.next_sel = reinterpret_cast<int*>(b); b += p.next_sel;
    L.next_slot = reinterpret_cast<int*>(b); b += p.next_slot;
    L.next_n = reinterpret_cast<int*>(b); b += p.next_n;
    L.next_commit = reinterpret_cast<int*>(b); b += p.next_commit;
    L.miss_flag = reinterpret_cast<uint8_t*>(b); b += p.mflag;
    L.scores = scores + (size_t)(l & 1) * (p.scores / 2 / sizeof(float));   // this layer's parity copy
    L.attn_part = part;
    L.attn_ml = ml;
    L.unit_done = done;
    L.score_done = done + d.U;
    L.host_k = L.host_v = nullptr;
    L.err = c->err;
    // slot pools start zeroed: rows past a context end that a tile still reads are then zeros
    // or earlier (finite) history rows, never uninitialised bit patterns
    cudaError_t e = cudaMemset(L.kpool, 0, p.kpool);
    if (e == cudaSuccess && L.vpool) e = cudaMemset(L.vpool, 0, p.vpool);
    if (e == cudaSuccess) e = cudaMemset(L.block2slot, 0xff, p.b2s);
    if (e == cudaSuccess) e = cudaMemset(L.slot2block, 0xff, p.s2b);
    if (e == cudaSuccess) e = cudaMemset(L.stamp, 0, p.stamp);
    if (e == cudaSuccess) e = cudaMemset(L.clock, 0, p.clock);
    if (e == cudaSuccess) e = cudaMemset(L.pend_n, 0xff, p.pend_n);
    if (e == cudaSuccess) e = cudaMemset(L.n_fetch, 0, p.nfetch);
    if (e == cudaSuccess) e = cudaMemset(L.next_commit, 0, p.next_commit);
    if (e != cudaSuccess) {
      delete c;
      return KVS_ERR_CUDA;
    }
  }
  if (cudaMemset(c->err, 0, p.err) != cudaSuccess || cudaMemset(done, 0, p.done) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    delete c;
    return KVS_ERR_CUDA;
  }
  if (attention_tma_supported(d)) {
    c->tmaps.resize(2 * (size_t)d.NL);
    const size_t rows = (size_t)d.U * d.C * d.bs;
    for (int l = 0; l < d.NL; ++l) {
      if (!make_pool_map(&c->tmaps[2 * l], c->layers[l].kpool, rows, d.dk, d.ebytes) ||
          !make_pool_map(&c->tmaps[2 * l + 1], c->layers[l].vpool, rows, d.dv, d.ebytes)) {
        c->tmaps.clear();
        break;
      }
    }
  }
  for (int l = 0; l < d.NL; ++l) {
    c->layers[l].tmK = c->tmaps.empty() ? nullptr : &c->tmaps[2 * l];
    c->layers[l].tmV = c->tmaps.empty() ? nullptr : &c->tmaps[2 * l + 1];
  }
  c->booted.assign(d.NL, 0);
  c->fetch_done.assign(d.NL, nullptr);
  c->fetch_pending.assign(d.NL, 0);
  c->sel_ready.assign(d.NL, nullptr);
  c->pf_done.assign(d.NL, nullptr);
  c->sel_pending.assign(d.NL, 0);
  c->pf_pending.assign(d.NL, 0);
  c->layer_start.assign(d.NL, nullptr);
  c->upd_done.assign(d.NL, nullptr);
  c->attn_done.assign(d.NL, nullptr);
  for (auto* v : {&c->sel_ready, &c->pf_done, &c->fetch_done, &c->layer_start, &c->upd_done, &c->attn_done})
    for (cudaEvent_t& ev : *v)
      if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
        ev = nullptr;
        kvs_destroy(c);
        return KVS_ERR_CUDA;
      }
  // the selection chain of overlapped lookahead steps is the step's critical path: highest priority
  int lo = 0, hi = 0;
  for (cudaStream_t& st : c->sel_stream)
    if (cudaDeviceGetStreamPriorityRange(&lo, &hi) != cudaSuccess ||
        cudaStreamCreateWithPriority(&st, cudaStreamNonBlocking, hi) != cudaSuccess) {
      st = nullptr;
      kvs_destroy(c);
      return KVS_ERR_CUDA;
    }
  *out = c;
  return KVS_OK;
}

kvs_status kvs_kernel_timer_arm(kvs_ctx* c, int kernel, int capacity) {
  if (!c || capacity < 0 || kernel < 1 || kernel > KVS_K_INDEX) return KVS_ERR_INVALID_ARG;
  kvs_ctx::Timer& t = c->timers[kernel];
  while ((int)t.start.size() < capacity) {
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess) return KVS_ERR_CUDA;
    if (cudaEventCreate(&b) != cudaSuccess) { cudaEventDestroy(a); return KVS_ERR_CUDA; }
    t.start.push_back(a);
    t.stop.push_back(b);
  }
  while ((int)t.start.size() > capacity) {
    cudaEventDestroy(t.start.back()); t.start.pop_back();
    cudaEventDestroy(t.stop.back()); t.stop.pop_back();
  }
  t.count = 0;
  return KVS_OK;
}

kvs_status kvs_kernel_timer_read(kvs_ctx* c, int kernel, double* total_ms, int* n_timed) {
  if (!c || !total_ms || !n_timed || kernel < 1 || kernel > KVS_K_INDEX) return KVS_ERR_INVALID_ARG;
  kvs_ctx::Timer& t = c->timers[kernel];
  double tot = 0.0;
  for (int i = 0; i < t.count; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(t.stop[i]) != cudaSuccess) return KVS_ERR_CUDA;
    if (cudaEventElapsedTime(&ms, t.start[i], t.stop[i]) != cudaSuccess) return KVS_ERR_CUDA;
    tot += ms;
  }
  *total_ms = tot;
  *n_timed = t.count;
  return KVS_OK;
}

unsigned long long kvs_launch_count(kvs_ctx* c) { return c ? c->launches : 0ull; }

kvs_status kvs_destroy(kvs_ctx* c) {
  if (!c) return KVS_ERR_INVALID_ARG;
  for (auto& t : c->timers) {
    for (cudaEvent_t e : t.start) cudaEventDestroy(e);
    for (cudaEvent_t e : t.stop) cudaEventDestroy(e);
  }
  for (auto* v : {&c->sel_ready, &c->pf_done, &c->fetch_done, &c->layer_start, &c->upd_done, &c->attn_done})
    for (cudaEvent_t e : *v)
      if (e) cudaEventDestroy(e);
  for (cudaStream_t st : c->sel_stream)
    if (st) cudaStreamDestroy(st);
  delete c;
  return KVS_OK;
}

kvs_status kvs_bind_host_kv(kvs_ctx* c, void* h_k, void* h_v) {
  if (!c || !h_k) return KVS_ERR_INVALID_ARG;
  if (c->d.v_shares_k ? h_v != nullptr : h_v == nullptr) return KVS_ERR_INVALID_ARG;
  void* dk = nullptr;
  void* dv = nullptr;
  // page-locked host memory only: where the device can also reach pageable memory (address
  // translation services), cudaHostGetDevicePointer alone would accept it
  for (void* h : {h_k, h_v}) {
    if (!h) continue;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, h) != cudaSuccess || a.type != cudaMemoryTypeHost) {
      cudaGetLastError();
      return KVS_ERR_HOST_MEM;
    }
  }
  if (cudaHostGetDevicePointer(&dk, h_k, 0) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_HOST_MEM;
  }
  if (h_v && cudaHostGetDevicePointer(&dv, h_v, 0) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_HOST_MEM;
  }
  c->host_k_dev = static_cast<const __nv_bfloat16*>(dk);
  c->host_v_dev = static_cast<const __nv_bfloat16*>(dv);
  const Dims& d = c->d;
  // touch every page once from the device: the first fetches then do not pay for translations
  const size_t rows = (size_t)d.NL * d.U * d.max_ctx;
  cudaError_t e = launch_touch_pages(dk, rows * d.dk * d.ebytes, c->err + 1, 0);
  if (e == cudaSuccess && dv) e = launch_touch_pages(dv, rows * d.dv * d.ebytes, c->err + 1, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return KVS_ERR_CUDA;
  for (int l = 0; l < d.NL; ++l) {
    size_t unit_rows = (size_t)d.U * d.max_ctx;
    // element offsets of bf16 pointers; E4M3 rows are half as many bytes
    c->layers[l].host_k = reinterpret_cast<const __nv_bfloat16*>(reinterpret_cast<const unsigned char*>(c->host_k_dev) +
                                                                 (size_t)l * unit_rows * d.dk * d.ebytes);
    c->layers[l].host_v = dv ? reinterpret_cast<const __nv_bfloat16*>(reinterpret_cast<const unsigned char*>(c->host_v_dev) +
                                                                      (size_t)l * unit_rows * d.dv * d.ebytes)
                             : nullptr;
  }
  return KVS_OK;
}

kvs_status kvs_index_build(kvs_ctx* c, int layer, void* d_index, const int* d_ctx_len, kvs_stream_t stream) {
  if (!layer_ok(c, layer) || !d_index || !d_ctx_len) return KVS_ERR_INVALID_ARG;
  if (!c->host_k_dev) return KVS_ERR_HOST_MEM;
  const Dims& d = c->d;
  __nv_bfloat16* idx = static_cast<__nv_bfloat16*>(d_index) + (size_t)layer * d.U * d.nb_max * d.didx;
  return cuda_status(timed(c, KVS_K_INDEX, S(stream), 1, [&] { return launch_index_build(d, c->layers[layer], idx, d_ctx_len, S(stream)); }));
}

kvs_status kvs_score_blocks(kvs_ctx* c, int layer, const void* d_score_q, int nq, const void* d_index,
                            const int* d_ctx_len, float* d_scores, kvs_stream_t stream) {
  if (!layer_ok(c, layer) || !d_score_q || !d_index || !d_ctx_len || !d_scores) return KVS_ERR_INVALID_ARG;
  const Dims& d = c->d;
  if (nq < 1 || nq > d.max_nq) return KVS_ERR_INVALID_ARG;
  if (!score_supported(d)) return KVS_ERR_NOT_SUPPORTED;
  const __nv_bfloat16* idx = static_cast<const __nv_bfloat16*>(d_index) + (size_t)layer * d.U * d.nb_max * d.didx;
  return cuda_status(timed(c, KVS_K_SCORE, S(stream), 1, [&] {
    return launch_score(d, idx, static_cast<const __nv_bfloat16*>(d_score_q), nq, d_ctx_len, d_scores, c->err, S(stream));
  }));
}

kvs_status kvs_topk_select(kvs_ctx* c, const float* d_scores, const int* d_ctx_len, int* d_sel, int* d_nsel,
                           kvs_stream_t stream) {
  if (!c || !d_scores || !d_ctx_len || !d_sel || !d_nsel) return KVS_ERR_INVALID_ARG;
  return cuda_status(timed(c, KVS_K_TOPK, S(stream), 1, [&] { return launch_topk(c->d, d_scores, d_ctx_len, d_sel, d_nsel, c->err, S(stream), c->tk[0].key ? &c->tk[0] : nullptr); }));
}

kvs_status kvs_cache_update(kvs_ctx* c, int layer, const int* d_sel, const int* d_nsel, const int* d_ctx_len,
                            int* d_slot_of_sel, const float* d_scores, kvs_stats* d_stats, kvs_stream_t stream) {
  if (!layer_ok(c, layer) || !d_sel || !d_nsel || !d_ctx_len || !d_slot_of_sel) return KVS_ERR_INVALID_ARG;
  if (c->d.evict_importance && !d_scores) return KVS_ERR_INVALID_ARG;
  if (!c->host_k_dev) return KVS_ERR_HOST_MEM;
  const Layer& L = c->layers[layer];
  cudaError_t e = timed(c, KVS_K_UPDATE, S(stream), 1, [&] {
    return launch_cache_update(c->d, L, d_sel, d_nsel, d_ctx_len, d_slot_of_sel,
                               c->d.evict_importance ? d_scores : nullptr, d_stats, S(stream));
  });
  if (e == cudaSuccess) e = timed(c, KVS_K_FETCH, S(stream), 1, [&] { return launch_fetch(c->d, L, d_ctx_len, S(stream)); });
  return cuda_status(e);
}

size_t kvs_snapshot_bytes(const kvs_config* cfg) {
  Dims d;
  if (!fill_dims(cfg, &d)) return 0;
  return snapshot_plan(d).total;
}

kvs_status kvs_cache_snapshot(kvs_ctx* c, int layer, void* d_snapshot, kvs_stream_t stream) {
  if (!layer_ok(c, layer) || !d_snapshot || (reinterpret_cast<uintptr_t>(d_snapshot) % kAlign)) return KVS_ERR_INVALID_ARG;
  const Dims& d = c->d;
  const Layer& L = c->layers[layer];
  const SnapshotPlan p = snapshot_plan(d);
  unsigned char* o = static_cast<unsigned char*>(d_snapshot);
  const size_t U = d.U;
  struct Part { void* dst; const void* src; size_t n; } parts[] = {
      {o, L.block2slot, U * d.nb_max * 4},
      {o + p.b2s, L.slot2block, U * d.C * 4},
      {o + p.b2s + p.s2b, L.stamp, U * d.C * 4},
      {o + p.b2s + p.s2b + p.stamp, L.clock, U * 4},
      {o + p.b2s + p.s2b + p.stamp + p.clock, L.pend_sel, U * d.Kb * 4},
      {o + p.b2s + p.s2b + p.stamp + p.clock + p.pend_sel, L.pend_slot, U * d.Kb * 4},
      {o + p.b2s + p.s2b + p.stamp + p.clock + p.pend_sel + p.pend_slot, L.pend_n, U * 4}};
  for (const Part& x : parts)
    if (cudaMemcpyAsync(x.dst, x.src, x.n, cudaMemcpyDeviceToDevice, S(stream)) != cudaSuccess) return KVS_ERR_CUDA;
  return KVS_OK;
}

kvs_status kvs_cache_restore(kvs_ctx* c, int layer, const void* d_snapshot, const int* d_ctx_len,
                             kvs_stream_t stream) {
  if (!layer_ok(c, layer) || !d_snapshot || !d_ctx_len || (reinterpret_cast<uintptr_t>(d_snapshot) % kAlign))
    return KVS_ERR_INVALID_ARG;
  if (!c->host_k_dev) return KVS_ERR_HOST_MEM;
  const Layer& L = c->layers[layer];
  cudaError_t e = timed(c, KVS_K_UPDATE, S(stream), 1, [&] {
    return launch_restore(c->d, L, static_cast<const unsigned char*>(d_snapshot), S(stream));
  });
  if (e == cudaSuccess) e = timed(c, KVS_K_FETCH, S(stream), 1, [&] { return launch_fetch(c->d, L, d_ctx_len, S(stream)); });
  return cuda_status(e);
}

kvs_status kvs_sparse_decode_attn(kvs_ctx* c, int layer, const void* d_q, const int* d_sel, const int* d_slot_of_sel,
                                  const int* d_nsel, const int* d_ctx_len, float* d_out, kvs_stream_t stream) {
  if (!layer_ok(c, layer) || !d_q || !d_sel || !d_slot_of_sel || !d_nsel || !d_ctx_len || !d_out)
    return KVS_ERR_INVALID_ARG;
  if (!attention_supported(c->d)) return KVS_ERR_NOT_SUPPORTED;
  return cuda_status(timed(c, KVS_K_ATTN, S(stream), attn_kernels(c->d), [&] {
    return launch_attention(c->d, c->layers[layer], static_cast<const __nv_bfloat16*>(d_q), d_sel, d_slot_of_sel, d_nsel,
                            d_ctx_len, d_out, S(stream));
  }));
}

kvs_status kvs_layer_prefetch(kvs_ctx* c, int dst_layer, const int* d_hint_sel, const int* d_hint_nsel,
                              const int* d_ctx_len, kvs_stats* d_stats, kvs_stream_t stream) {
  if (!layer_ok(c, dst_layer) || dst_layer < 1 || !d_hint_sel || !d_hint_nsel || !d_ctx_len)
    return KVS_ERR_INVALID_ARG;
  if (!c->host_k_dev) return KVS_ERR_HOST_MEM;
  const Layer& L = c->layers[dst_layer];
  cudaError_t e = cudaSuccess;
  // the hint is the layer below's selection of this step: wait for its top-K when that ran on
  // another stream
  if (c->sel_pending[dst_layer - 1]) e = cudaStreamWaitEvent(S(stream), c->sel_ready[dst_layer - 1], 0);
  if (e == cudaSuccess)
    e = timed(c, KVS_K_PREFETCH, S(stream), 1, [&] {
      return launch_prefetch(c->d, L, d_hint_sel, d_hint_nsel, d_ctx_len, d_stats, S(stream));
    });
  if (e == cudaSuccess) e = timed(c, KVS_K_FETCH, S(stream), 1, [&] { return launch_fetch(c->d, L, d_ctx_len, S(stream)); });
  // the destination layer's next update waits for this
  if (e == cudaSuccess) e = cudaEventRecord(c->pf_done[dst_layer], S(stream));
  if (e == cudaSuccess) c->pf_pending[dst_layer] = 1;
  return cuda_status(e);
}

kvs_status kvs_advance_ctx(kvs_ctx* c, int* d_ctx_len, kvs_stream_t stream) {
  if (!c || !d_ctx_len) return KVS_ERR_INVALID_ARG;
  return cuda_status(timed(c, 0, S(stream), 1, [&] { return launch_advance(c->d.B, d_ctx_len, S(stream)); }));
}

kvs_status kvs_append(kvs_ctx* c, int layer, const void* d_k_new, const void* d_v_new, void* d_index,
                      const int* d_ctx_len, kvs_stream_t stream) {
  if (!layer_ok(c, layer) || !d_k_new || !d_index || !d_ctx_len) return KVS_ERR_INVALID_ARG;
  if (!c->d.v_shares_k && !d_v_new) return KVS_ERR_INVALID_ARG;
  if (!aligned16(d_k_new) || !aligned16(d_v_new)) return KVS_ERR_INVALID_ARG;
  if (!c->host_k_dev) return KVS_ERR_HOST_MEM;
  const Dims& d = c->d;
  __nv_bfloat16* idx = static_cast<__nv_bfloat16*>(d_index) + (size_t)layer * d.U * d.nb_max * d.didx;
  return cuda_status(timed(c, KVS_K_APPEND, S(stream), 1, [&] {
    return launch_append(d, c->layers[layer], static_cast<const __nv_bfloat16*>(d_k_new),
                         static_cast<const __nv_bfloat16*>(d_v_new), idx, d_ctx_len, S(stream));
  }));
}

kvs_status kvs_decode_step(kvs_ctx* c, int layer, const void* d_q, const void* d_score_q, int nq,
                           const void* d_k_new, const void* d_v_new, void* d_index, const int* d_ctx_len,
                           float* d_out, kvs_stats* d_stats, int* d_sel_out, int* d_nsel_out, kvs_stream_t stream,
                           kvs_stream_t copy_stream) {
  if (!layer_ok(c, layer) || !d_q || !d_index || !d_ctx_len || !d_out) return KVS_ERR_INVALID_ARG;
  if (!c->host_k_dev) return KVS_ERR_HOST_MEM;
  const Dims& d = c->d;
  if (!score_supported(d) || !attention_supported(d)) return KVS_ERR_NOT_SUPPORTED;
  if (d_score_q == nullptr) nq = 1;
  if (nq < 1 || nq > d.max_nq) return KVS_ERR_INVALID_ARG;
  if (d_k_new && !d.v_shares_k && !d_v_new) return KVS_ERR_INVALID_ARG;
  if (!aligned16(d_k_new) || !aligned16(d_v_new)) return KVS_ERR_INVALID_ARG;
  cudaStream_t s = S(stream);
  cudaStream_t cs = copy_stream ? S(copy_stream) : s;
  Layer& L = c->layers[layer];
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(d_q);
  const __nv_bfloat16* sq = d_score_q ? static_cast<const __nv_bfloat16*>(d_score_q) : q;
  __nv_bfloat16* idx = static_cast<__nv_bfloat16*>(d_index) + (size_t)layer * d.U * d.nb_max * d.didx;
  int* sel = d_sel_out ? d_sel_out : L.sel;
  int* nsel = d_nsel_out ? d_nsel_out : L.nsel;
  cudaError_t e = cudaSuccess;
  const __nv_bfloat16* kn = static_cast<const __nv_bfloat16*>(d_k_new);
  const __nv_bfloat16* vn = static_cast<const __nv_bfloat16*>(d_v_new);
  // the selection chain (score, top-K, update) runs on `ss`: `s`, or in lookahead mode with a copy
  // stream the context's own selection stream, beside the attention on `s`
  cudaStream_t ss = s;
  auto score = [&](const __nv_bfloat16* rows, int n) {
    return timed(c, KVS_K_SCORE, ss, 1, [&] { return launch_score(d, idx, rows, n, d_ctx_len, L.scores, c->err, ss); });
  };
  auto topk = [&](int* so, int* no) {
    const kvs::TopkScratch* tks = c->tk[layer & 1].key ? &c->tk[layer & 1] : nullptr;
    cudaError_t r = timed(c, KVS_K_TOPK, ss, 1, [&] { return launch_topk(d, L.scores, d_ctx_len, so, no, c->err, ss, tks); });
    if (r == cudaSuccess) r = cudaEventRecord(c->sel_ready[layer], ss);   // hint for a prefetch into layer + 1
    if (r == cudaSuccess) c->sel_pending[layer] = 1;
    return r;
  };
  auto update = [&](const int* so, const int* no) {
    cudaError_t r = cudaSuccess;
    if (c->pf_pending[layer]) {       // a prefetch into this layer ran on another stream
      r = cudaStreamWaitEvent(ss, c->pf_done[layer], 0);
      c->pf_pending[layer] = 0;
    }
    if (r != cudaSuccess) return r;
    return timed(c, KVS_K_UPDATE, ss, 1,
                 [&] { return launch_cache_update(d, L, so, no, d_ctx_len, L.slot_of_sel,
                                                  d.evict_importance ? L.scores : nullptr, d_stats, ss); });
  };
  // top-K then update on the same selection: one fused kernel when the unit's scores fit a CTA's
  // shared memory, else the two kernels
  auto select = [&](int* so, int* no) {
    if (!select_update_fusable(d)) {
      cudaError_t r = topk(so, no);
      return r == cudaSuccess ? update(so, no) : r;
    }
    cudaError_t r = cudaSuccess;
    if (c->pf_pending[layer]) {       // a prefetch into this layer ran on another stream
      r = cudaStreamWaitEvent(ss, c->pf_done[layer], 0);
      c->pf_pending[layer] = 0;
    }
    if (r == cudaSuccess)
      r = timed(c, KVS_K_UPDATE, ss, 1, [&] {
        return launch_select_update(d, L, L.scores, d_ctx_len, so, no, L.slot_of_sel, d_stats, ss);
      });
    if (r == cudaSuccess) r = cudaEventRecord(c->sel_ready[layer], ss);   // hint for a prefetch into layer + 1
    if (r == cudaSuccess) c->sel_pending[layer] = 1;
    return r;
  };
  auto fetch = [&](cudaStream_t fs) {
    return timed(c, KVS_K_FETCH, fs, 1, [&] { return launch_fetch(d, L, d_ctx_len, fs); });
  };
  auto attn = [&](const int* so, const int* slots, const int* no) {
    return timed(c, KVS_K_ATTN, s, attn_kernels(d),
                 [&] { return launch_attention(d, L, q, so, slots, no, d_ctx_len, d_out, s); });
  };
  if (kn) e = timed(c, KVS_K_APPEND, s, 1, [&] { return launch_append(d, L, kn, vn, idx, d_ctx_len, s); });
  if (!d.lookahead) {
    if (e == cudaSuccess) e = score(sq, nq);
    if (e == cudaSuccess) e = select(sel, nsel);
    if (cs == s || !attention_tma_supported(d) || !L.tmK || !L.tmV) {
      if (e == cudaSuccess) e = fetch(s);
      if (e == cudaSuccess) e = attn(sel, L.slot_of_sel, nsel);
      return cuda_status(e);
    }
    // with a copy stream: the misses are fetched there while the attention runs over the hits
    // (their slots are resident), then the attention over the fetched blocks merges both parts
    if (e == cudaSuccess) e = cudaEventRecord(c->upd_done[layer], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, c->upd_done[layer], 0);
    if (e == cudaSuccess) e = fetch(cs);
    if (e == cudaSuccess) e = cudaEventRecord(c->fetch_done[layer], cs);
    for (int phase = 1; phase <= 2 && e == cudaSuccess; ++phase) {
      if (phase == 2) e = cudaStreamWaitEvent(s, c->fetch_done[layer], 0);
      if (e == cudaSuccess)
        e = timed(c, KVS_K_ATTN, s, 1, [&] {
          return launch_attention_tma(d, L, L.tmK, L.tmV, q, sel, L.slot_of_sel, nsel, d_ctx_len, d_out, s, phase);
        });
    }
    return cuda_status(e);
  }
  // no selection yet (the layer's first lookahead step): pick S_t from the current query and make
  // it resident, on the stream that runs the selection chain, before the attention reads it
  auto bootstrap = [&](cudaStream_t fs) {
    cudaError_t r = score(q, 1);
    if (r == cudaSuccess) r = select(L.sel, L.nsel);
    if (r == cudaSuccess) r = fetch(fs);
    if (r == cudaSuccess) c->booted[layer] = 1;
    return r;
  };
  if (cs == s) {
    // one stream: attention over S_t, then the selection of S_{t+1} and its fetch
    if (e == cudaSuccess && !c->booted[layer]) e = bootstrap(s);
    if (e == cudaSuccess) e = attn(L.pend_sel, L.pend_slot, L.pend_n);
    if (e == cudaSuccess) e = score(sq, nq);
    if (e == cudaSuccess) e = select(sel, nsel);
    if (e == cudaSuccess) e = fetch(s);
    return cuda_status(e);
  }
  // Overlapped: the selection of S_{t+1} (score with the drafts, top-K, update with S_t pinned,
  // which stages the new pending selection) starts on the selection stream as soon as the layer
  // below has finished its attention, and runs beside this layer's attention over S_t on `s`.  The
  // fetch waits for both: it writes only slots the update freed, and it commits the staged
  // selection, which the attention must no longer be reading.  Layers of one parity share the
  // block-score and top-K scratch, so their chains run on the same one of the two selection streams.
  ss = c->sel_stream[layer & 1];
  if (layer_kernel_supported(d, nq, L.tmK && L.tmV)) {
    // one kernel on `s` runs this layer's attention over S_t beside the selection of S_{t+1} (a
    // fixed split of one wave of CTAs); the fetch then waits for it on the copy stream
    if (e == cudaSuccess && !c->booted[layer]) {
      // the bootstrap's selection chain runs on the selection stream after the work queued on `s`
      // (the inputs), and `s` waits for it
      e = cudaEventRecord(c->layer_start[layer], s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(ss, c->layer_start[layer], 0);
      if (e == cudaSuccess) e = bootstrap(ss);
      if (e == cudaSuccess) e = cudaEventRecord(c->upd_done[layer], ss);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s, c->upd_done[layer], 0);
    }
    if (e == cudaSuccess)
      e = timed(c, KVS_K_ATTN, s, 1,
                [&] { return launch_layer(d, L, q, idx, sq, nq, d_ctx_len, d_out, sel, nsel, d_stats, s); });
    if (e == cudaSuccess) e = cudaEventRecord(c->sel_ready[layer], s);   // hint for a prefetch into layer + 1
    if (e == cudaSuccess) c->sel_pending[layer] = 1;
    if (e == cudaSuccess) e = cudaEventRecord(c->attn_done[layer], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, c->attn_done[layer], 0);
    if (e == cudaSuccess) e = fetch(cs);
    if (e == cudaSuccess) e = cudaEventRecord(c->fetch_done[layer], cs);
    if (e == cudaSuccess) c->fetch_pending[layer] = 1;
    return cuda_status(e);
  }
  if (e == cudaSuccess) e = cudaEventRecord(c->layer_start[layer], s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ss, c->layer_start[layer], 0);
  if (e == cudaSuccess && !c->booted[layer]) {
    e = bootstrap(ss);
    if (e == cudaSuccess) e = cudaEventRecord(c->upd_done[layer], ss);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, c->upd_done[layer], 0);
  }
  if (e == cudaSuccess) e = score(sq, nq);
  if (e == cudaSuccess) e = select(sel, nsel);
  if (e == cudaSuccess) e = cudaEventRecord(c->upd_done[layer], ss);
  if (e == cudaSuccess) e = attn(L.pend_sel, L.pend_slot, L.pend_n);
  if (e == cudaSuccess) e = cudaEventRecord(c->attn_done[layer], s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, c->attn_done[layer], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, c->upd_done[layer], 0);
  if (e == cudaSuccess) e = fetch(cs);
  if (e == cudaSuccess) e = cudaEventRecord(c->fetch_done[layer], cs);
  if (e == cudaSuccess) c->fetch_pending[layer] = 1;
  return cuda_status(e);
}

kvs_status kvs_join(kvs_ctx* c, kvs_stream_t stream) {
  if (!c) return KVS_ERR_INVALID_ARG;
  for (int l = 0; l < c->d.NL; ++l) {
    if (c->fetch_pending[l]) {
      if (cudaStreamWaitEvent(S(stream), c->fetch_done[l], 0) != cudaSuccess) return KVS_ERR_CUDA;
      c->fetch_pending[l] = 0;
    }
    if (c->pf_pending[l]) {
      if (cudaStreamWaitEvent(S(stream), c->pf_done[l], 0) != cudaSuccess) return KVS_ERR_CUDA;
      c->pf_pending[l] = 0;
    }
    c->sel_pending[l] = 0;
  }
  return KVS_OK;
}

kvs_status kvs_cache_export(kvs_ctx* c, int layer, int* h_block2slot, int* h_slot2block, unsigned* h_stamp,
                            unsigned* h_clock) {
  if (!layer_ok(c, layer)) return KVS_ERR_INVALID_ARG;
  const Dims& d = c->d;
  const Layer& L = c->layers[layer];
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess && h_block2slot)
    e = cudaMemcpy(h_block2slot, L.block2slot, (size_t)d.U * d.nb_max * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && h_slot2block)
    e = cudaMemcpy(h_slot2block, L.slot2block, (size_t)d.U * d.C * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && h_stamp) e = cudaMemcpy(h_stamp, L.stamp, (size_t)d.U * d.C * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && h_clock) e = cudaMemcpy(h_clock, L.clock, (size_t)d.U * 4, cudaMemcpyDeviceToHost);
  return cuda_status(e);
}

kvs_status kvs_slot_pools(kvs_ctx* c, int layer, void** d_k_pool, void** d_v_pool) {
  if (!layer_ok(c, layer) || !d_k_pool || !d_v_pool) return KVS_ERR_INVALID_ARG;
  *d_k_pool = c->layers[layer].kpool;
  *d_v_pool = c->layers[layer].vpool;
  return KVS_OK;
}

kvs_status kvs_poll_error(kvs_ctx* c, kvs_status* device_status) {
  if (!c || !device_status) return KVS_ERR_INVALID_ARG;
  unsigned v = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&v, c->err, sizeof(v), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(c->err, 0, sizeof(v));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  *device_status = static_cast<kvs_status>(v);
  return cuda_status(e);
}

}  // extern "C"
