// Decode attention over the selected cache slots: the TMA kernel (the CTA's work is in
// kvs_attn_tma.cuh) and its launcher.
#include "kvs_attn_tma.cuh"

namespace kvs {

using namespace tma;

namespace {

template <int NT, bool FP8>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    attn_tma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, Dims d,
                    Layer L, const __nv_bfloat16* __restrict__ q, const int* __restrict__ sel,
                    const int* __restrict__ slot_of_sel, const int* __restrict__ nsel,
                    const int* __restrict__ ctx_len, float* __restrict__ out, Plan plan) {
  extern __shared__ unsigned char smem_raw[];
  attn_tma_cta<NT, FP8>(tmK, tmV, d, L, q, sel, slot_of_sel, nsel, ctx_len, out, plan, blockIdx.x, smem_raw);
}

int sm_count() { return device_sm_count(); }

}  // namespace

int attention_tma_supported(const Dims& d) {
  return !d.v_shares_k && d.dk == D && d.dv == D && d.G <= 16 && d.bs % 16 == 0;
}

// Partial-result slots per unit the TMA path needs (one per CTA segment of a unit, for each of the
// two phases of a split launch).
int attention_tma_partials(const Dims& d) { return 2 * make_plan(d, sm_count()).max_segs; }

cudaError_t launch_attention_tma(const Dims& d, const Layer& L, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                 const __nv_bfloat16* q, const int* sel, const int* slot_of_sel, const int* nsel,
                                 const int* ctx_len, float* out, cudaStream_t s, int phase) {
  Plan plan = make_plan(d, sm_count());
  plan.phase = phase;
  auto go = [&](auto kern, int smem) {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(plan.n_cta), dim3(kThreads), (size_t)smem, s, *tmK, *tmV, d, L, q, sel, slot_of_sel,
                      nsel, ctx_len, out, plan);
  };
  cudaError_t e;
  if (d.fp8)
    e = d.G <= 8 ? go(attn_tma_kernel<1, true>, Smem<1, true>::bytes(d.G, plan.per_cta))
                 : go(attn_tma_kernel<2, true>, Smem<2, true>::bytes(d.G, plan.per_cta));
  else
    e = d.G <= 8 ? go(attn_tma_kernel<1, false>, Smem<1, false>::bytes(d.G, plan.per_cta))
                 : go(attn_tma_kernel<2, false>, Smem<2, false>::bytes(d.G, plan.per_cta));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvs
