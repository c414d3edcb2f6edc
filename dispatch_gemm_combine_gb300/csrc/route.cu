// Top-k routing of router logits: the step before the expert layer.
//
// One warp per token.  Lane l holds the token's logits of experts
// l, l + 32, l + 64, ... (E <= 1024, so at most 32 per lane) in registers.
// Each of the k rounds picks the largest logit not yet chosen: every lane
// proposes its own best (the lowest id among equal values, since a lane's
// ids increase with the register index), a butterfly reduction keeps the
// larger value, or the lower id when the values are equal, and the owning
// lane marks the expert as taken.  Lane j keeps choice j; the weights are a
// softmax over the k chosen logits, normalised by their maximum (choice 0).
#include <cfloat>

#include "kernels.h"

namespace moe {

namespace {

constexpr int kMaxPerLane = 32;   // E <= 1024

__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int64_t T,
                                                    int E, int k, int* __restrict__ topk_idx,
                                                    float* __restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int nloc = (E + 31) >> 5;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       t < T; t += warps) {
    const float* row = logits + t * E;
    float v[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      v[i] = (i < nloc && e < E) ? __ldg(row + e) : 0.f;
    }
    uint32_t taken = 0;   // bit i: expert lane + 32 i is chosen (or does not exist)
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
      if (i >= nloc || lane + 32 * i >= E) taken |= 1u << i;
    int my_id = 0;
    float my_v = 0.f;
    for (int j = 0; j < k; ++j) {
      float best = -FLT_MAX;
      int bid = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        if (!((taken >> i) & 1u) && (bid == 0x7fffffff || v[i] > best)) {
          best = v[i];
          bid = lane + 32 * i;
        }
      }
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, d);
        const int oid = __shfl_xor_sync(0xffffffffu, bid, d);
        if (ob > best || (ob == best && oid < bid)) {
          best = ob;
          bid = oid;
        }
      }
      if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
      if (lane == j) {
        my_id = bid;
        my_v = best;
      }
    }
    const float m = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = (lane < k) ? expf(my_v - m) : 0.f;
    float sum = ex;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
    if (lane < k) {
      topk_idx[t * k + lane] = my_id;
      topk_w[t * k + lane] = ex / sum;
    }
  }
}

}  // namespace

cudaError_t launch_route(const float* logits, int64_t T, int E, int k, int* topk_idx,
                         float* topk_w, int num_sms, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (E > 32 * kMaxPerLane || k > 32 || k > E) return cudaErrorInvalidValue;
  int64_t blocks = (T + 7) / 8;
  if (blocks > static_cast<int64_t>(num_sms) * 16) blocks = static_cast<int64_t>(num_sms) * 16;
  route_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(logits, T, E, k, topk_idx, topk_w);
  return cudaGetLastError();
}

}  // namespace moe
