// bf16 backward data-gradient grouped GEMMs: down dgrad + activation
// backward + d(topk weights) partials, gate_up dgrad.
#include "gemm.cuh"

namespace moe {

cudaError_t launch_gemm_bf16_dgrad(int mode, const GemmMaps& maps, const GemmArgs& a, int sms,
                                   cudaStream_t st) {
  using T = __nv_bfloat16;
  switch (mode) {
    case kDgradDown:
      return a.gu_interleaved ? launch_gemm_t<T, kDgradDown, 256, 3, true>(maps, a, sms, st)
                              : launch_gemm_t<T, kDgradDown, 256, 3>(maps, a, sms, st);
    case kDgradGateUp: return launch_gemm_t<T, kDgradGateUp, 256, 6, false, true>(maps, a, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
