// fp32-storage instantiation of every grouped GEMM mode (TF32 tensor-core
// products with fp32 accumulation).
#include "gemm.cuh"

namespace moe {

cudaError_t launch_gemm_f32(int mode, const GemmMaps& maps, const GemmArgs& a, int sms,
                            cudaStream_t st) {
  using T = float;
  switch (mode) {
    case kFwdGateUp: return launch_gemm_t<T, kFwdGateUp, 256, 4>(maps, a, sms, st);
    case kFwdDown: return launch_gemm_t<T, kFwdDown, 256, 4>(maps, a, sms, st);
    case kDgradDown:   // (the TF32 gate_up forward reads either layout through strided views)
      return a.gu_interleaved ? launch_gemm_t<T, kDgradDown, 256, 3, true>(maps, a, sms, st)
                              : launch_gemm_t<T, kDgradDown, 256, 3>(maps, a, sms, st);
    case kDgradGateUp: return launch_gemm_t<T, kDgradGateUp, 256, 4>(maps, a, sms, st);
    case kWgradDown: return launch_gemm_t<T, kWgradDown, 256, 4>(maps, a, sms, st);
    case kWgradGateUp: return launch_gemm_t<T, kWgradGateUp, 256, 3>(maps, a, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
