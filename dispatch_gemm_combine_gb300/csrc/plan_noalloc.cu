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
#include <cudaTypedefs.h>

#include <mutex>

#include "abi_internal.h"
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

// Device address of g_plan_scratch.  In host code the symbol names a
// host-side stand-in, never the device array, so the address is resolved
// with cudaGetSymbolAddress, with the device current.  It is resolved once
// per device context: the cache remembers the CUDA driver's unique id of the
// context it was resolved in, and a call that finds another context current
// (after cudaDeviceReset, the module and its array are loaded anew) resolves
// it again instead of using a stale address.
struct ScratchAddr {
  bool done = false;
  unsigned long long ctx_id = 0;
  int* ptr = nullptr;
};
std::mutex g_mu;
ScratchAddr g_addr[64];

struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxFns& ctx_fns() {
  static CtxFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return f;
}

// Unique id of the current context; false if there is none yet (or the
// driver cannot say), in which case the address is resolved afresh.
bool current_ctx_id(unsigned long long* id) {
  const CtxFns& f = ctx_fns();
  if (!f.get_current || !f.get_id) return false;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return f.get_id(ctx, id) == CUDA_SUCCESS;
}

moe_status scratch_for_current_device(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchAddr& a = g_addr[dev];
  unsigned long long id = 0;
  const bool have_id = current_ctx_id(&id);
  if (!a.done || !have_id || id != a.ctx_id) {
    void* p = nullptr;
    // (this also creates the device's context if no runtime call has yet)
    if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    a.ptr = static_cast<int*>(p);
    a.done = current_ctx_id(&a.ctx_id);   // not cached when the context has no id
  }
  *out = a.ptr;
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_plan_noalloc(const moe_shape* s, const int32_t* topk_idx,
                                       const moe_plan_t* plan, moe_stream_t stream) {
  // the same argument rules as moe_plan, minus the workspace
  if (!abi_shape_ok(s) || !plan || !plan->counts || !plan->offsets) return MOE_ERR_INVALID_ARG;
  const int64_t Tk = s->T * static_cast<int64_t>(s->k);
  if (Tk > 0 && (!topk_idx || !plan->perm || !plan->inv)) return MOE_ERR_INVALID_ARG;
  // the fixed scratch bounds the problem size: ceil(T*k / 1024) * E ints
  if (plan_blkhist_ints(Tk, s->E) > static_cast<size_t>(kHistInts)) return MOE_ERR_WORKSPACE;
  int sms = 0;
  const moe_status ds = abi_device_sms(&sms);
  if (ds != MOE_OK) return ds;
  int* scratch = nullptr;
  const moe_status st0 = scratch_for_current_device(&scratch);
  if (st0 != MOE_OK) return st0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The error word must start at zero on every call; the histograms and the
  // padded offsets are fully rewritten by the kernels.
  if (abi_tracked_memset(scratch + kErrOff, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
  if (abi_tracked_plan(topk_idx, Tk, s->E, plan->counts, plan->offsets, plan->perm, plan->inv,
                       scratch + kPoffOff, scratch + kHistOff, scratch + kErrOff,
                       st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
