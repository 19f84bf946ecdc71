// Block selection for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or have torch allocate for them): code that runs inside
// an allocator hook, where re-entering the allocator deadlocks, plug-ins that live in a process
// whose device memory is fully budgeted by another runtime, or embedded deployments that forbid
// allocation after start-up.  (It makes CUDA API calls itself, so it must not be called from a
// stream callback or a cudaLaunchHostFunc host function.)  kvs_select_blocks_noalloc serves them: it
// scores and selects one layer's blocks (the same kernels as kvs_score_blocks followed by
// kvs_topk_select) with the block scores kept in the file-scope device array below, so the
// caller passes only its inputs and outputs.  The array (KVS_NOALLOC_MAX_SCORES floats) is held
// by every GPU that loads the library, until the process exits.
#include <mutex>

#include "kvs_common.cuh"

static __device__ __align__(256) float kvs_noalloc_scores[KVS_NOALLOC_MAX_SCORES];
static __device__ __align__(256) unsigned kvs_noalloc_status[64];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
float* g_scores_ptr[kMaxDevices] = {};
unsigned* g_status_ptr[kMaxDevices] = {};

// Device addresses of the two arrays on the current device, looked up once per device.  In host
// code the arrays' names are host-side stand-ins, never device addresses.
bool scratch_of_current_device(float** scores, unsigned** status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scores_ptr[dev]) {
    void* p = nullptr;
    void* q = nullptr;
    if (cudaGetSymbolAddress(&p, kvs_noalloc_scores) != cudaSuccess || !p) return false;
    if (cudaGetSymbolAddress(&q, kvs_noalloc_status) != cudaSuccess || !q) return false;
    g_scores_ptr[dev] = static_cast<float*>(p);
    g_status_ptr[dev] = static_cast<unsigned*>(q);
  }
  *scores = g_scores_ptr[dev];
  *status = g_status_ptr[dev];
  return true;
}

}  // namespace

namespace kvs {
bool config_to_dims(const kvs_config* c, Dims* d);
}

extern "C" kvs_status kvs_select_blocks_noalloc(const kvs_config* cfg, const void* d_score_q, int nq,
                                                const void* d_index_layer, const int* d_ctx_len, int* d_sel,
                                                int* d_nsel, unsigned* d_status, kvs_stream_t stream) {
  kvs::Dims d;
  if (!kvs::config_to_dims(cfg, &d)) return KVS_ERR_INVALID_ARG;
  // the size limit first, so an oversized shape is refused whatever else is passed
  if ((long long)d.U * d.nb_max > (long long)KVS_NOALLOC_MAX_SCORES) return KVS_ERR_CAPACITY;
  if (!d_score_q || !d_index_layer || !d_ctx_len || !d_sel || !d_nsel) return KVS_ERR_INVALID_ARG;
  if (nq < 1 || nq > d.max_nq) return KVS_ERR_INVALID_ARG;
  if (!kvs::score_supported(d)) return KVS_ERR_NOT_SUPPORTED;
  float* scores = nullptr;
  unsigned* status = nullptr;
  if (!scratch_of_current_device(&scores, &status)) return KVS_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned* err = d_status ? d_status : status;
  cudaError_t e = kvs::launch_score(d, static_cast<const __nv_bfloat16*>(d_index_layer),
                                    static_cast<const __nv_bfloat16*>(d_score_q), nq, d_ctx_len, scores, err, s);
  if (e == cudaSuccess) e = kvs::launch_topk(d, scores, d_ctx_len, d_sel, d_nsel, err, s, nullptr);
  return e == cudaSuccess ? KVS_OK : KVS_ERR_CUDA;
}
