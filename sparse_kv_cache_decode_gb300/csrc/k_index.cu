// Block summaries (the mean key, or the per-dimension [max | min] of the keys) and the per-step
// append of one token.
#include <math.h>

#include <algorithm>

#include "kvs_common.cuh"
#include "kvs_ptx.cuh"

namespace kvs {

// One warp per block: lanes own 4 consecutive dims at a time; tokens are summed in fp32 one at
// a time in ascending position, divided by the present-token count (IEEE) and rounded to bf16
// (round-to-nearest-even).  Bound mode keeps the running max and min instead (strict compares,
// so among equal values the earliest token's is kept) and writes [max | min].
template <int CHUNKS>  // 4-dim chunks per lane = ceil(dk / 128)
__global__ void __launch_bounds__(256) index_build_kernel(Dims d, Layer L, __nv_bfloat16* __restrict__ index,
                                                          const int* __restrict__ ctx_len) {
  const int u = blockIdx.y;
  const int r = u / d.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * 8 + warp;
  const int len = ctx_len[r];
  if (len < 0 || len > d.max_ctx) {
    if (threadIdx.x == 0) set_error(L.err, KVS_ERR_BAD_INDEX);
    return;
  }
  const int nb = n_blocks_of(len, d.bs);
  if (b >= nb) return;
  const int t0 = b * d.bs, t1 = min(t0 + d.bs, len);
  const int nchunk = d.dk / 4;
  const __nv_bfloat16* rows = L.host_k + (size_t)u * d.max_ctx * d.dk;
  // E4M3 history: byte rows, each code widened to fp32(decode(code) * k_scale)
  const unsigned char* rows8 = reinterpret_cast<const unsigned char*>(L.host_k) + (size_t)u * d.max_ctx * d.dk;
  float acc[CHUNKS][4], mx[CHUNKS][4], mn[CHUNKS][4];
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[c][e] = 0.f;
  for (int t = t0; t < t1; ++t) {
    const uint2* row = reinterpret_cast<const uint2*>(rows + (size_t)t * d.dk);
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
      int ch = lane + 32 * c;
      if (ch < nchunk) {
        float x[4];
        if (d.fp8) {
          const uint32_t c4 = *reinterpret_cast<const uint32_t*>(rows8 + (size_t)t * d.dk + ch * 4);
#pragma unroll
          for (int e = 0; e < 4; ++e) x[e] = __fmul_rn(e4m3_to_f32((c4 >> (8 * e)) & 255u), d.k_scale);
        } else {
          const uint2 v = row[ch];
          x[0] = bf16_lo(v.x);
          x[1] = bf16_hi(v.x);
          x[2] = bf16_lo(v.y);
          x[3] = bf16_hi(v.y);
        }
        if (d.bound) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (t == t0 || x[e] > mx[c][e]) mx[c][e] = x[e];
            if (t == t0 || x[e] < mn[c][e]) mn[c][e] = x[e];
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[c][e] = __fadd_rn(acc[c][e], x[e]);
        }
      }
    }
  }
  const float n = (float)(t1 - t0);
  uint2* out = reinterpret_cast<uint2*>(index + ((size_t)u * d.nb_max + b) * d.didx);
  if (d.bound) {   // the kept values are bf16 already: packing them is exact
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
      int ch = lane + 32 * c;
      if (ch < nchunk) {
        out[ch] = make_uint2(pack_bf16x2(mx[c][0], mx[c][1]), pack_bf16x2(mx[c][2], mx[c][3]));
        out[nchunk + ch] = make_uint2(pack_bf16x2(mn[c][0], mn[c][1]), pack_bf16x2(mn[c][2], mn[c][3]));
      }
    }
    return;
  }
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) {
    int ch = lane + 32 * c;
    if (ch < nchunk) {
      uint2 o;
      o.x = pack_bf16x2(__fdiv_rn(acc[c][0], n), __fdiv_rn(acc[c][1], n));
      o.y = pack_bf16x2(__fdiv_rn(acc[c][2], n), __fdiv_rn(acc[c][3], n));
      out[ch] = o;
    }
  }
}

cudaError_t launch_index_build(const Dims& d, const Layer& L, __nv_bfloat16* index, const int* ctx_len,
                               cudaStream_t s) {
  dim3 grid((d.nb_max + 7) / 8, d.U);
  int chunks = (d.dk / 4 + 31) / 32;
  if (chunks <= 1) index_build_kernel<1><<<grid, 256, 0, s>>>(d, L, index, ctx_len);
  else if (chunks <= 2) index_build_kernel<2><<<grid, 256, 0, s>>>(d, L, index, ctx_len);
  else if (chunks <= 5) index_build_kernel<5><<<grid, 256, 0, s>>>(d, L, index, ctx_len);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

// One CTA per unit.  Writes the token at position len-1 to the host history and, when its block
// is resident, to the block's slot (16-byte vectors); then recomputes the block's index key from
// its present tokens, in token order, taking the new token's values from k_new and the earlier
// rows from the block's slot when it is resident (the same bf16 values as the host rows, read
// from HBM instead of over the host link), else from the host history.
__global__ void __launch_bounds__(128) append_kernel(Dims d, Layer L, const __nv_bfloat16* __restrict__ k_new,
                                                     const __nv_bfloat16* __restrict__ v_new,
                                                     __nv_bfloat16* __restrict__ index,
                                                     const int* __restrict__ ctx_len) {
  kvs_pdl_entry();
  const int u = blockIdx.x;
  const int r = u / d.Hkv;
  const int len = ctx_len[r];
  if (len < 1 || len > d.max_ctx) {
    if (threadIdx.x == 0) set_error(L.err, KVS_ERR_BAD_INDEX);
    return;
  }
  const int p = len - 1;
  const int b = p / d.bs, row_in_blk = p - b * d.bs;
  const int slot = L.block2slot[(size_t)u * d.nb_max + b];
  if (d.fp8) {
    // quantise the token (round to nearest even, saturating), store the codes in the history and
    // the resident slot, then rebuild the block's key from the stored values
    uint16_t* hk = reinterpret_cast<uint16_t*>(const_cast<__nv_bfloat16*>(L.host_k)) +
                   (((size_t)u * d.max_ctx + p) * d.dk) / 2;
    uint16_t* sk = slot >= 0 ? reinterpret_cast<uint16_t*>(L.kpool) + ((((size_t)u * d.C + slot) * d.bs + row_in_blk) * d.dk) / 2
                             : nullptr;
    for (int i = threadIdx.x; i < d.dk / 2; i += blockDim.x) {
      const float a = __bfloat162float(k_new[(size_t)u * d.dk + 2 * i]);
      const float c = __bfloat162float(k_new[(size_t)u * d.dk + 2 * i + 1]);
      const uint16_t code = (uint16_t)f32x2_to_e4m3x2(__fdiv_rn(a, d.k_scale), __fdiv_rn(c, d.k_scale));
      hk[i] = code;
      if (sk) sk[i] = code;
    }
    uint16_t* hv = reinterpret_cast<uint16_t*>(const_cast<__nv_bfloat16*>(L.host_v)) +
                   (((size_t)u * d.max_ctx + p) * d.dv) / 2;
    uint16_t* sv = slot >= 0 ? reinterpret_cast<uint16_t*>(L.vpool) + ((((size_t)u * d.C + slot) * d.bs + row_in_blk) * d.dv) / 2
                             : nullptr;
    for (int i = threadIdx.x; i < d.dv / 2; i += blockDim.x) {
      const float a = __bfloat162float(v_new[(size_t)u * d.dv + 2 * i]);
      const float c = __bfloat162float(v_new[(size_t)u * d.dv + 2 * i + 1]);
      const uint16_t code = (uint16_t)f32x2_to_e4m3x2(__fdiv_rn(a, d.v_scale), __fdiv_rn(c, d.v_scale));
      hv[i] = code;
      if (sv) sv[i] = code;
    }
    const unsigned char* rows8 =
        slot >= 0 ? reinterpret_cast<const unsigned char*>(L.kpool) + ((size_t)u * d.C + slot) * d.bs * d.dk
                  : reinterpret_cast<const unsigned char*>(L.host_k) + ((size_t)u * d.max_ctx + (size_t)b * d.bs) * d.dk;
    const float n = (float)(row_in_blk + 1);
    for (int i = threadIdx.x; i < d.dk; i += blockDim.x) {
      float acc = 0.f;
      for (int t = 0; t < row_in_blk; ++t) acc = __fadd_rn(acc, __fmul_rn(e4m3_to_f32(rows8[(size_t)t * d.dk + i]), d.k_scale));
      const float kn = __bfloat162float(k_new[(size_t)u * d.dk + i]);
      const uint32_t code = f32x2_to_e4m3x2(__fdiv_rn(kn, d.k_scale), 0.f) & 255u;
      acc = __fadd_rn(acc, __fmul_rn(e4m3_to_f32(code), d.k_scale));
      index[((size_t)u * d.nb_max + b) * d.didx + i] = __float2bfloat16_rn(__fdiv_rn(acc, n));
    }
    return;
  }
  {
    uint4* hk = reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(L.host_k) + ((size_t)u * d.max_ctx + p) * d.dk);
    const uint4* kn = reinterpret_cast<const uint4*>(k_new + (size_t)u * d.dk);
    uint4* sk = slot >= 0 ? reinterpret_cast<uint4*>(L.kpool + (((size_t)u * d.C + slot) * d.bs + row_in_blk) * d.dk)
                          : nullptr;
    for (int i = threadIdx.x; i < d.dk / 8; i += blockDim.x) {
      const uint4 x = kn[i];
      hk[i] = x;
      if (sk) sk[i] = x;
    }
  }
  if (!d.v_shares_k) {
    uint4* hv = reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(L.host_v) + ((size_t)u * d.max_ctx + p) * d.dv);
    const uint4* vn = reinterpret_cast<const uint4*>(v_new + (size_t)u * d.dv);
    uint4* sv = slot >= 0 ? reinterpret_cast<uint4*>(L.vpool + (((size_t)u * d.C + slot) * d.bs + row_in_blk) * d.dv)
                          : nullptr;
    for (int i = threadIdx.x; i < d.dv / 8; i += blockDim.x) {
      const uint4 x = vn[i];
      hv[i] = x;
      if (sv) sv[i] = x;
    }
  }
  // summary of block b over tokens [b*bs, len): earlier rows in token order, then the new one
  const __nv_bfloat16* rows = slot >= 0 ? L.kpool + ((size_t)u * d.C + slot) * d.bs * d.dk
                                        : L.host_k + ((size_t)u * d.max_ctx + (size_t)b * d.bs) * d.dk;
  const int nt = row_in_blk;                                // earlier rows of the block
  const float n = (float)(nt + 1);
  if (d.bound) {
    for (int i = threadIdx.x; i < d.dk; i += blockDim.x) {
      float mx = 0.f, mn = 0.f;
      for (int t = 0; t <= nt; ++t) {
        const float x = __bfloat162float(t < nt ? rows[(size_t)t * d.dk + i] : k_new[(size_t)u * d.dk + i]);
        if (t == 0 || x > mx) mx = x;
        if (t == 0 || x < mn) mn = x;
      }
      __nv_bfloat16* o = index + ((size_t)u * d.nb_max + b) * d.didx;
      o[i] = __float2bfloat16_rn(mx);
      o[d.dk + i] = __float2bfloat16_rn(mn);
    }
    return;
  }
  for (int i = threadIdx.x; i < d.dk; i += blockDim.x) {
    float acc = 0.f;
    int t = 0;
    for (; t + 8 <= nt; t += 8) {
      float x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = __bfloat162float(rows[(size_t)(t + j) * d.dk + i]);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc = __fadd_rn(acc, x[j]);
    }
    for (; t < nt; ++t) acc = __fadd_rn(acc, __bfloat162float(rows[(size_t)t * d.dk + i]));
    acc = __fadd_rn(acc, __bfloat162float(k_new[(size_t)u * d.dk + i]));
    index[((size_t)u * d.nb_max + b) * d.didx + i] = __float2bfloat16_rn(__fdiv_rn(acc, n));
  }
}

cudaError_t launch_append(const Dims& d, const Layer& L, const __nv_bfloat16* k_new, const __nv_bfloat16* v_new,
                          __nv_bfloat16* index, const int* ctx_len, cudaStream_t s) {
  launch_pdl(append_kernel, dim3(d.U), dim3(128), 0, s, d, L, k_new, v_new, index, ctx_len);
  return cudaGetLastError();
}

// One 16-byte read per 4 KiB page of a mapped host range, so the device's translations of the
// whole history exist before the first decode step fetches from it.  The loaded words are folded
// into *sink only to keep the loads.
__global__ void __launch_bounds__(256) touch_pages_kernel(const uint4* __restrict__ base, size_t n_pages,
                                                          unsigned* sink) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  unsigned acc = 0;
  for (size_t p = (size_t)blockIdx.x * blockDim.x + threadIdx.x; p < n_pages; p += stride) {
    uint4 v = base[p * 256];  // 4096 / 16
    acc ^= v.x ^ v.w;
  }
  if (acc == 0x9e3779b9u) atomicAdd(sink, 1u);
}

cudaError_t launch_touch_pages(const void* base, size_t bytes, unsigned* sink, cudaStream_t s) {
  size_t n_pages = bytes / 4096;
  if (n_pages == 0) return cudaSuccess;
  touch_pages_kernel<<<4 * 152, 256, 0, s>>>(static_cast<const uint4*>(base), n_pages, sink);
  return cudaGetLastError();
}

__global__ void advance_kernel(int B, int* ctx_len) {
  kvs_pdl_entry();
  int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r < B) ctx_len[r] += 1;
}

// E4M3 codes of bf16 values: 8 per thread (one 16-byte load, one 8-byte store), the tail one by one.
__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const __nv_bfloat16* __restrict__ src, uint8_t* __restrict__ dst,
                                                            size_t n, float scale) {
  const size_t n8 = n / 8;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint4 v = reinterpret_cast<const uint4*>(src)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(w[2 * h]), scale), __fdiv_rn(bf16_hi(w[2 * h]), scale));
      const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(w[2 * h + 1]), scale), __fdiv_rn(bf16_hi(w[2 * h + 1]), scale));
      out[h] = lo | (hi << 16);
    }
    reinterpret_cast<uint2*>(dst)[i] = make_uint2(out[0], out[1]);
  }
  for (size_t i = n8 * 8 + (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = (uint8_t)(f32x2_to_e4m3x2(__fdiv_rn(__bfloat162float(src[i]), scale), 0.f) & 255u);
}

cudaError_t launch_advance(int B, int* ctx_len, cudaStream_t s) {
  launch_pdl(advance_kernel, dim3((B + 127) / 128), dim3(128), 0, s, B, ctx_len);
  return cudaGetLastError();
}

}  // namespace kvs

extern "C" kvs_status kvs_quantize_e4m3(const void* d_src_bf16, void* d_dst, size_t n, float scale, kvs_stream_t stream) {
  if (!d_src_bf16 || !d_dst || !(scale > 0.f) || isinf(scale)) return KVS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(d_src_bf16) & 15u) || (reinterpret_cast<uintptr_t>(d_dst) & 7u)) return KVS_ERR_INVALID_ARG;
  if (n == 0) return KVS_OK;
  const size_t n8 = n / 8 + 1;
  const int blocks = (int)std::min<size_t>((n8 + 255) / 256, 4096);
  kvs::quantize_e4m3_kernel<<<blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(d_src_bf16), static_cast<uint8_t*>(d_dst), n, scale);
  return cudaGetLastError() == cudaSuccess ? KVS_OK : KVS_ERR_CUDA;
}
