// bf16 forward grouped GEMMs: gate_up + activation, down + routing weight.
#include "gemm.cuh"

namespace moe {

cudaError_t launch_gemm_bf16_fwd(int mode, const GemmMaps& maps, const GemmArgs& a, int sms,
                                 cudaStream_t st) {
  using T = __nv_bfloat16;
  switch (mode) {
    case kFwdGateUp:
      return a.gu_interleaved ? launch_gemm_t<T, kFwdGateUp, 256, 6, true>(maps, a, sms, st)
                              : launch_gemm_t<T, kFwdGateUp, 256, 6, false, true>(maps, a, sms, st);
    case kFwdDown: return launch_gemm_t<T, kFwdDown, 256, 6, false, true>(maps, a, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
