// moe_plan_noalloc: the dispatch plan without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the moment they need a plan:
// code that runs inside an allocator-free region (a custom memory pool that
// is already carved up, a real-time path where cudaMalloc's implicit device
// synchronisation is not acceptable, or an embedding runtime that owns all
// device memory and hands out only the tensors it manages).  For them the
// plan kernels' scratch (per-chunk expert histograms, the tile-padded
// offsets and an error word) lives in a fixed array in this library's device
// image instead of in a workspace.  The array exists once per GPU that loads
// the library and stays allocated until the process exits.
#include <mutex>

#include "kernels.h"
#include "moe.h"

namespace {

using namespace moe;

// Scratch layout (ints): [0, 64) error word and padding, [64, 64 + 2112)
// padded offsets and tile-pair prefix (2 * (E + 1) <= 2050), then the
// per-chunk histograms.
constexpr int kScratchInts = 1 << 18;   // 1 MiB
constexpr int kErrOff = 0;
constexpr int kPoffOff = 64;
constexpr int kHistOff = kPoffOff + 2112;
constexpr int kHistInts = kScratchInts - kHistOff;

static __device__ __align__(256) int g_plan_scratch[kScratchInts];

// Device address of g_plan_scratch, resolved once per device with that
// device current.  Host code must not use the symbol itself as a pointer.
struct ScratchAddr {
  bool done = false;
  int* ptr = nullptr;
};
std::mutex g_mu;
ScratchAddr g_addr[64];

moe_status scratch_for_current_device(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchAddr& a = g_addr[dev];
  if (!a.done) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    a.ptr = static_cast<int*>(p);
    a.done = true;
  }
  *out = a.ptr;
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_plan_noalloc(const moe_shape* s, const int32_t* topk_idx,
                                       const moe_plan_t* plan, moe_stream_t stream) {
  if (!s || !plan || !plan->counts || !plan->offsets) return MOE_ERR_INVALID_ARG;
  if (s->T < 0 || s->k < 1 || s->k > 32 || s->E < s->k || s->E > 1024) return MOE_ERR_INVALID_ARG;
  const int64_t Tk = s->T * static_cast<int64_t>(s->k);
  if (Tk >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
  if (Tk > 0 && (!topk_idx || !plan->perm || !plan->inv)) return MOE_ERR_INVALID_ARG;
  // the fixed scratch bounds the problem size: ceil(T*k / 1024) * E ints
  if (plan_blkhist_ints(Tk, s->E) > static_cast<size_t>(kHistInts)) return MOE_ERR_WORKSPACE;
  int major = 0, minor = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;
  int* scratch = nullptr;
  const moe_status st0 = scratch_for_current_device(&scratch);
  if (st0 != MOE_OK) return st0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The error word must start at zero on every call; the histograms and the
  // padded offsets are fully rewritten by the kernels.
  if (cudaMemsetAsync(scratch + kErrOff, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_plan(topk_idx, Tk, s->E, plan->counts, plan->offsets, plan->perm, plan->inv,
                  scratch + kPoffOff, scratch + kHistOff, scratch + kErrOff, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
