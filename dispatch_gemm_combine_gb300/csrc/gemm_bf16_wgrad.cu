// bf16 per-expert weight-gradient GEMMs (fp32 outputs).  The computed
// operand (w*a for the down weights, dH1 for gate_up) is a bf16 hi/lo pair.
#include "gemm.cuh"

namespace moe {

cudaError_t launch_gemm_bf16_wgrad(int mode, const GemmMaps& maps, const GemmArgs& a, int sms,
                                   cudaStream_t st) {
  using T = __nv_bfloat16;
  switch (mode) {
    case kWgradDown: return launch_gemm_t<T, kWgradDown, 256, 6>(maps, a, sms, st);
    case kWgradGateUp: return launch_gemm_t<T, kWgradGateUp, 256, 6>(maps, a, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
