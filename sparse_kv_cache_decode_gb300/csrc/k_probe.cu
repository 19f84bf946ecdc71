// Host-link read probe (diagnostics): SM zero-copy reads of items from device-mapped host memory,
// the access pattern of the block fetch without its slot writes, so that the link's best read
// rate for that pattern can be measured beside a copy-engine transfer.
#include "kvs_common.cuh"

namespace kvs {
namespace {

constexpr int kProbeUnroll = 16;

// One item per warp at a time; each lane keeps up to 16 16-byte loads in flight.  The loaded
// words are folded into one value per thread, and a thread stores only when that value equals a
// sentinel, so the loads stay live without writing HBM.  Offsets outside the region are skipped
// and counted in sink[1].
__global__ void host_read_probe_kernel(const uint4* __restrict__ base, unsigned long long region_bytes,
                                       const long long* __restrict__ offsets, int n_items, int item_vecs,
                                       unsigned* sink) {
  const int lane = threadIdx.x & 31;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const unsigned long long item_bytes = (unsigned long long)item_vecs * 16ull;
  unsigned acc = 0;
  for (int it = gwarp; it < n_items; it += nwarps) {
    const long long off = offsets[it];
    if (off < 0 || (off & 15) || (unsigned long long)off + item_bytes > region_bytes) {
      if (lane == 0) atomicAdd(sink + 1, 1u);
      continue;
    }
    const uint4* p = base + off / 16;
    for (int v0 = 0; v0 < item_vecs; v0 += 32 * kProbeUnroll) {
      uint4 x[kProbeUnroll];
#pragma unroll
      for (int k = 0; k < kProbeUnroll; ++k) {
        const int v = v0 + k * 32 + lane;
        x[k] = v < item_vecs ? p[v] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < kProbeUnroll; ++k) acc ^= x[k].x ^ x[k].y ^ x[k].z ^ x[k].w;
    }
  }
  if (acc == 0x9e3779b9u) atomicAdd(sink, 1u);
}

}  // namespace
}  // namespace kvs

extern "C" kvs_status kvs_probe_host_read(const void* h_base, size_t region_bytes, const long long* d_offsets,
                                          int n_items, int item_bytes, int n_ctas, int threads, unsigned* d_sink,
                                          kvs_stream_t stream) {
  if (!h_base || !d_offsets || !d_sink || n_items < 0 || item_bytes < 16 || (item_bytes % 16) || n_ctas < 1 ||
      n_ctas > 65535 || threads < 32 || threads > 1024 || (threads % 32))
    return KVS_ERR_INVALID_ARG;
  void* dev = nullptr;
  if (cudaHostGetDevicePointer(&dev, const_cast<void*>(h_base), 0) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_HOST_MEM;
  }
  if (n_items == 0) return KVS_OK;
  kvs::host_read_probe_kernel<<<n_ctas, threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(dev), (unsigned long long)region_bytes, d_offsets, n_items, item_bytes / 16, d_sink);
  return cudaGetLastError() == cudaSuccess ? KVS_OK : KVS_ERR_CUDA;
}
