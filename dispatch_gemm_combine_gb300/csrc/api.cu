// C ABI of the MoE expert layer: argument checks, workspace layout, TMA
// descriptor encoding and the launch sequence of each entry point.
//
// Forward  (token-repeat page: repeat, masked expert FFN, weighted sum):
//   plan -> gather X into tile-padded expert-grouped rows Xp
//        -> gate_up GEMM, activation fused in the epilogue (A, saved H1)
//        -> down GEMM, routing weight fused in the epilogue (Ow, reusing Xp)
//        -> k-way combine per token (the dispatch-and-combine page's
//           index_add_ step, in a fixed order).
// Backward (backward page: d hidden_states, topk_weights, gate/up/down):
//   gather dY, X -> down dgrad + activation backward (dH1, Aw, dw partials)
//   -> dw reduce -> down wgrad -> gate_up dgrad (dXp, reusing dYp)
//   -> combine dXp into dX -> gate_up wgrad.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "abi_internal.h"
#include "kernels.h"
#include "moe.h"

namespace moe {

cudaError_t launch_gemm_bf16_fwd(int, const GemmMaps&, const GemmArgs&, int, cudaStream_t);
cudaError_t launch_gemm_bf16_dgrad(int, const GemmMaps&, const GemmArgs&, int, cudaStream_t);
cudaError_t launch_gemm_bf16_wgrad(int, const GemmMaps&, const GemmArgs&, int, cudaStream_t);
cudaError_t launch_gemm_f32(int, const GemmMaps&, const GemmArgs&, int, cudaStream_t);

cudaError_t launch_gemm(int mode, int elem_bytes, const GemmMaps& maps, const GemmArgs& args,
                        int num_sms, cudaStream_t st) {
  if (elem_bytes == 4) return launch_gemm_f32(mode, maps, args, num_sms, st);
  switch (mode) {
    case kFwdGateUp:
    case kFwdDown: return launch_gemm_bf16_fwd(mode, maps, args, num_sms, st);
    case kDgradDown:
    case kDgradGateUp: return launch_gemm_bf16_dgrad(mode, maps, args, num_sms, st);
    default: return launch_gemm_bf16_wgrad(mode, maps, args, num_sms, st);
  }
}

// Output-column tile width of each mode (must match the instantiations).
int gemm_block_n(int mode, int elem_bytes) {
  if (mode == kFwdGateUp) return 128;
  return 256;
}

// Output rows per weight-gradient m-tile (one CTA's rows).
int gemm_block_m(int mode, int elem_bytes) {
  (void)mode;
  (void)elem_bytes;
  return 128;
}

// Rows of the K-major weight box of a dgrad: the bf16 gate_up dgrad runs as
// CTA pairs, each holding half of the 256 columns.
uint32_t dgrad_b_rows(int mode, int elem_bytes) {
  return (mode == kDgradGateUp && elem_bytes == 2) ? 128 : 256;
}

}  // namespace moe

using namespace moe;

namespace {

constexpr int kMaxExperts = 1024;
// Effective row count (sum w^2)^2 / sum w^4 of an expert from which its bf16
// weight gradients take the computed operand (dH1, w*a) as one bf16 value
// instead of a bf16 hi + lo pair.  The rounding error of a single bf16
// operand, relative to the expert gradient's rms, falls with the rows that
// carry weight: simulated on the layer's workload distributions (clamped GLU
// and SwiGLU, weights N(0, 0.02), fan-in and N(0, 0.3), routing weights of
// softmaxes over 4 and 8 logits), the largest element error stays at or below
// 0.022 rms from n_eff = 150 up, and rises to 0.03 - 0.05 rms below
// n_eff = 30.  Below this count the pair is kept (error ~1e-4 rms).
constexpr float kSplitMinNeff = 160.f;
constexpr int kMaxTopK = 32;
std::atomic<uint64_t> g_timeout_ns{2000000000ull};

// ------------------------------------------------------------ launch accounting
// Kernel kinds, for the launch counter and the optional event timer.
enum Kind : int {
  kKPlan = 0, kKOffsets, kKGather, kKFwdGateUp, kKFwdDown, kKCombine, kKDgradDown, kKDwReduce,
  kKWgradDown, kKDgradGateUp, kKWgradGateUp, kKMemset, kKTranspose, kKRoute, kKBiasDot,
  kKBiasGrad, kKSplitSelect, kKGatherIndex, kKCombineDense, kNumKinds
};
const char* const kKindNames[kNumKinds] = {
    "plan", "padded_offsets", "gather_rows", "gemm_fwd_gate_up_act", "gemm_fwd_down_scale",
    "combine", "gemm_dgrad_down_act_bwd", "dw_reduce", "gemm_wgrad_down", "gemm_dgrad_gate_up",
    "gemm_wgrad_gate_up", "memset", "transpose_f32", "route", "bias_slot_dot", "bias_colsum",
    "split_select", "gather_index", "combine_dense"};

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_profile{0};
struct ProfRec {
  int kind;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
std::vector<ProfRec> g_prof_pending;
std::vector<cudaEvent_t> g_event_pool;
double g_prof_ms[kNumKinds];
uint64_t g_prof_n[kNumKinds];

cudaEvent_t pool_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Run one launcher, counting its kernels and, when the timer is on,
// bracketing it with events on the launching stream.
template <typename F>
cudaError_t tracked(int kind, int nkernels, cudaStream_t st, F&& launch) {
  cudaEvent_t a = nullptr, b = nullptr;
  if (g_profile.load(std::memory_order_relaxed)) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    a = pool_event();
    b = pool_event();
    if (a && b) cudaEventRecord(a, st);
  }
  const cudaError_t e = launch();
  g_launches.fetch_add(static_cast<uint64_t>(nkernels), std::memory_order_relaxed);
  if (a && b) {
    cudaEventRecord(b, st);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_pending.push_back({kind, a, b});
  }
  return e;
}

// ------------------------------------------------------------ device cache
struct DevInfo {
  bool init = false;
  bool supported = false;
  int sms = 0;
};
std::mutex g_mu;
DevInfo g_dev[64];

moe_status device_info(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.sms = n;
    d.init = true;
  }
  if (!d.supported) return MOE_ERR_UNSUPPORTED;
  *sms = d.sms;
  return MOE_OK;
}

// ------------------------------------------------------------ TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

CUtensorMapDataType tma_dtype(int es) {
  return es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
}

// 2-D map over a row-major [rows, cols] view with row stride `ld` elements.
bool map2d(CUtensorMap* m, int es, const void* base, uint64_t cols, uint64_t rows, uint64_t ld,
           uint32_t box_c, uint32_t box_r, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * es};
  cuuint32_t box[2] = {box_c, box_r};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, tma_dtype(es), 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over [d2, d1, d0] with strides (elements) s1 for d1 and s2 for d2.
bool map3d(CUtensorMap* m, int es, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
           uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1 * es, s2 * es};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, tma_dtype(es), 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Epilogue output view: element (b, r, c) at p[b*bstride + r*ld + c],
// written only for r < rows and c < cols.
OutDesc out_view(const void* p, int64_t ld, int64_t rows, int64_t cols, int64_t bstride = 0) {
  OutDesc o;
  o.ptr = const_cast<void*>(p);
  o.ld = ld;
  o.bstride = bstride;
  o.rows = static_cast<int>(rows);
  o.cols = static_cast<int>(cols);
  return o;
}

// ------------------------------------------------------------ shape & layout
int elem_bytes(const moe_shape* s) { return s->dtype == MOE_FP32 ? 4 : 2; }

bool shape_ok(const moe_shape* s) {
  if (!s) return false;
  if (s->T < 0 || s->H < 8 || s->I < 8 || (s->H % 8) || (s->I % 8)) return false;
  if (s->k < 1 || s->k > kMaxTopK || s->E < s->k || s->E > kMaxExperts) return false;
  if (s->act != MOE_ACT_SWIGLU && s->act != MOE_ACT_CLAMPED_GLU) return false;
  if (s->dtype != MOE_BF16 && s->dtype != MOE_FP32) return false;
  if (s->gate_up_layout != MOE_GATE_UP_CONCAT && s->gate_up_layout != MOE_GATE_UP_INTERLEAVED)
    return false;
  if (s->out_fp32 != 0 && s->out_fp32 != 1) return false;
  if (s->T * static_cast<int64_t>(s->k) >= (1ll << 31)) return false;
  return true;
}

// Upper bound on the rows of the tile-padded expert-grouped layout:
// sum_e ceil(M_e / 128) * 128 with sum M_e = Tk and at most min(E, Tk)
// experts holding a row.
int64_t rows_max(const moe_shape* s) {
  const int64_t Tk = s->T * s->k;
  const int64_t live = Tk < s->E ? Tk : s->E;
  return (Tk + live * (kRowTile - 1)) / kRowTile * kRowTile;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct Layout {
  size_t err = 0, counts = 0, offsets = 0, perm = 0, inv = 0, poff = 0, blkhist = 0;
  size_t xp = 0, act = 0, ow = 0, dyp = 0, dh1 = 0, dh1lo = 0, aw = 0, awlo = 0, dxp = 0;
  size_t dwpart = 0, h1 = 0, lo_flags = 0;
  // fp32 storage only: K-major copies for the TF32 products
  size_t wguT = 0, wdT = 0, awT = 0, dypT = 0, xpT = 0, dh1T = 0, wdR = 0, wguR = 0;
  size_t total = 0;
};

int dgrad_down_ntiles(const moe_shape* s) { return (s->I + 255) / 256; }

// The context saved by the training forward: the expert-grouped token rows
// Xp [rows_max, H] in the storage dtype, then (256-byte aligned) the fp32
// gate | up pre-activations [rows_max, 2I].
size_t saved_rows(const moe_shape* s) {
  const size_t r = static_cast<size_t>(rows_max(s));
  return r > 0 ? r : 1;
}
size_t saved_h1_offset(const moe_shape* s) {
  return align256(saved_rows(s) * s->H * elem_bytes(s));
}
// The saved pre-activations are fp16 for the clamped GLU with bf16 storage
// when fp16 represents the clamp limit exactly and |L| <= 32768 (values past
// the clamp become markers, values inside stay inside, so the backward's
// clamp masks are exact), fp32 otherwise.
bool h1_half(const moe_shape* s) {
  if (elem_bytes(s) != 2 || s->act != MOE_ACT_CLAMPED_GLU) return false;
  const float L = s->clamp_limit;
  if (!(L >= -32768.f && L <= 32768.f)) return false;
  return __half2float(__float2half_rn(L)) == L;
}
size_t h1_elem_bytes(const moe_shape* s) { return h1_half(s) ? 2 : 4; }

Layout layout(const moe_shape* s, int which) {
  Layout L;
  const int64_t Tk = s->T * s->k;
  const int64_t R = rows_max(s);
  const size_t es = elem_bytes(s);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L.err = take(256);
  L.poff = take(sizeof(int) * 2 * (s->E + 1));   // padded offsets, then tile-pair prefix
  if (which == 0 || which == 1) L.blkhist = take(sizeof(int) * plan_blkhist_ints(Tk, s->E));
  if (which == 1) {
    L.counts = take(sizeof(int) * s->E);
    L.offsets = take(sizeof(int) * (s->E + 1));
    L.perm = take(sizeof(int) * (Tk > 0 ? Tk : 1));
    L.inv = take(sizeof(int) * (Tk > 0 ? Tk : 1));
    L.xp = take(es * R * s->H);
    L.act = take(es * R * s->I);
    L.ow = take(sizeof(float) * R * s->H);
    if (es == 4) {
      L.wguT = take(sizeof(float) * s->E * 2ull * s->I * s->H);
      L.wdT = take(sizeof(float) * s->E * static_cast<size_t>(s->I) * s->H);
    }
  }
  if (which == 2 || which == 3) {
    L.dyp = take(es * R * s->H);
    L.dh1 = take(es * R * 2 * s->I);
    L.aw = take(es * R * s->I);
    if (es == 2) {  // bf16 remainders of dH1 and w*a (operands of the weight gradients)
      L.dh1lo = take(es * R * 2 * s->I);
      L.awlo = take(es * R * s->I);
    } else {
      L.awT = take(es * R * s->I);
      L.dypT = take(es * R * s->H);
      L.xpT = take(es * R * s->H);
      L.dh1T = take(es * R * 2 * s->I);
      L.wdR = take(sizeof(float) * s->E * static_cast<size_t>(s->I) * s->H);
      L.wguR = take(sizeof(float) * s->E * 2ull * s->I * s->H);
    }
    L.dxp = take(sizeof(float) * R * s->H);
    // one partial per 256-column tile of the down dgrad, then the b_down term
    L.dwpart = take(sizeof(float) * R * (dgrad_down_ntiles(s) + 1));
    L.lo_flags = take(sizeof(int) * s->E);
  }
  if (which == 3) {   // backward without a saved context: recompute it
    L.xp = take(es * R * s->H);
    L.h1 = take(h1_elem_bytes(s) * R * 2 * s->I);
    if (es == 4) L.wguT = take(sizeof(float) * s->E * 2ull * s->I * s->H);
  }
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// The optional biases with a NULL struct read as "all NULL"; every pointer
// that is given must be 16-byte aligned.
moe_bias_t bias_or_none(const moe_bias_t* b) {
  moe_bias_t z;
  std::memset(&z, 0, sizeof(z));
  return b ? *b : z;
}
bool bias_aligned(const moe_bias_t& b) {
  auto ok = [](const void* p) { return !p || aligned16(p); };
  return ok(b.b_gate_up) && ok(b.b_down) && ok(b.db_gate_up) && ok(b.db_down);
}

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

#define MOE_CUDA(x)                             \
  do {                                          \
    if ((x) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

GemmArgs base_args(const moe_shape* s, const int* poff, const int* counts, const int* offsets,
                   const int* perm, const float* w, int* err) {
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.poff = poff;
  a.counts = counts;
  a.offsets = offsets;
  a.perm = perm;
  a.topk_w = w;
  a.tk = static_cast<int>(s->T * s->k);
  a.E = s->E;
  a.act = s->act;
  a.gu_interleaved = s->gate_up_layout == MOE_GATE_UP_INTERLEAVED ? 1 : 0;
  a.limit = s->clamp_limit;
  a.alpha = s->alpha;
  a.I = s->I;
  a.rows_max = rows_max(s);
  a.h1_half = h1_half(s) ? 1 : 0;
  a.err = err;
  a.timeout_ns = g_timeout_ns.load();
  return a;
}

// gate_up GEMM (+ the optional bias b_gate_up) + activation on the grouped
// rows xp: the activation into aact [R, I] and, when h1 is given, the fp32
// pre-activations [R, 2I] (gate | up).  fp32 storage first transposes the
// weights into wguT.
moe_status enqueue_gate_up(const moe_shape* s, const void* xp, const void* w_gate_up,
                           const void* b_gate_up, float* wguT,
                           void* aact, void* h1, int* poff, const int* counts,
                           const int* offsets, const int* perm, const float* topk_w, int* err,
                           int sms, cudaStream_t st) {
  const int es = elem_bytes(s);
  const int64_t R = rows_max(s);
  const int H = s->H, I = s->I, E = s->E;
  const uint32_t BK = 128 / es, CH = 128 / es;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  const char* wgu = static_cast<const char*>(w_gate_up);
  GemmMaps m1;
  const uint32_t AROWS = 128;
  const bool il = s->gate_up_layout == MOE_GATE_UP_INTERLEAVED;
  bool ok = map2d(&m1.a, es, xp, H, R, H, BK, AROWS, SW);
  if (es == 2 && il) {
    // interleaved columns: one view of all 2I columns (the kernel loads the
    // gate/up pairs of its outputs as consecutive columns)
    ok = ok && map3d(&m1.b0, es, wgu, 2ll * I, H, E, 2ll * I, 2ll * I * H, CH, BK, SW);
    m1.b1 = m1.b0;
  } else if (es == 2) {
    ok = ok && map3d(&m1.b0, es, wgu, I, H, E, 2ll * I, 2ll * I * H, CH, BK, SW) &&
         map3d(&m1.b1, es, wgu + static_cast<size_t>(I) * es, I, H, E, 2ll * I, 2ll * I * H, CH,
               BK, SW);
  } else {
    // TF32 takes K-major operands only: use the transposed weights [E, 2I, H];
    // gate rows are [0, I) (concatenated) or the even rows (interleaved)
    MOE_CUDA(tracked(kKTranspose, 1, st, [&] {
      return launch_transpose_f32(static_cast<const float*>(w_gate_up), wguT, E, H, 2 * I, st);
    }));
    const int64_t rstride = il ? 2ll * H : H;
    const size_t up0 = il ? static_cast<size_t>(H) : static_cast<size_t>(I) * H;
    ok = ok && map3d(&m1.b0, es, wguT, H, I, E, rstride, 2ll * I * H, BK, 128, SW) &&
         map3d(&m1.b1, es, wguT + up0, H, I, E, rstride, 2ll * I * H, BK, 128, SW);
  }
  if (!ok) return MOE_ERR_CUDA;
  m1.a2 = m1.a;
  // bf16 with concatenated columns tiles tokens on the MMA's N side; short
  // units use a 32-row box
  if (es == 2 && !il && !map2d(&m1.a2, es, xp, H, R, H, BK, 32, SW)) return MOE_ERR_CUDA;
  GemmArgs a1 = base_args(s, poff, counts, offsets, perm, topk_w, err);
  a1.out[0] = out_view(aact, I, R, I);
  if (h1) {
    a1.out[1] = out_view(h1, 2ll * I, R, I);
    a1.out[2] = out_view(static_cast<char*>(h1) + h1_elem_bytes(s) * I, 2ll * I, R, I);
  }
  a1.num_kb = (H + BK - 1) / BK;
  a1.n_tiles = (I + gemm_block_n(kFwdGateUp, es) - 1) / gemm_block_n(kFwdGateUp, es);
  a1.save_h1 = h1 ? 1 : 0;
  a1.bias = b_gate_up;
  MOE_CUDA(tracked(kKFwdGateUp, 1, st, [&] { return launch_gemm(kFwdGateUp, es, m1, a1, sms, st); }));
  return MOE_OK;
}

}  // namespace

// ------------------------------------------------------------ shared with other ABI units
namespace moe {

bool abi_shape_ok(const moe_shape* s) { return shape_ok(s); }

moe_status abi_device_sms(int* sms) { return device_info(sms); }

cudaError_t abi_tracked_plan(const int* idx, int64_t Tk, int E, int* counts, int* offsets,
                             int* perm, int* inv, int* poff, int* blkhist, int* err,
                             cudaStream_t st) {
  return tracked(kKPlan, Tk > 0 ? 3 : 1, st, [&] {
    return launch_plan(idx, Tk, E, counts, offsets, perm, inv, poff, blkhist, err, st);
  });
}

cudaError_t abi_tracked_memset(void* p, int value, size_t bytes, cudaStream_t st) {
  return tracked(kKMemset, 1, st, [&] { return cudaMemsetAsync(p, value, bytes, st); });
}

}  // namespace moe

// ====================================================================== ABI
extern "C" {

size_t moe_workspace_size(const moe_shape* shape, int which) {
  if (!shape_ok(shape) || which < 0 || which > 3) return 0;
  return layout(shape, which).total;
}

size_t moe_saved_size(const moe_shape* shape) {
  if (!shape_ok(shape)) return 0;
  return saved_h1_offset(shape) + saved_rows(shape) * 2 * shape->I * h1_elem_bytes(shape);
}

uint64_t moe_set_wait_timeout_ns(uint64_t ns) { return g_timeout_ns.exchange(ns); }

uint64_t moe_kernel_launch_count(void) { return g_launches.load(); }

int moe_profile_enable(int on) { return g_profile.exchange(on ? 1 : 0); }

const char* moe_profile_kernel_name(int kind) {
  return (kind >= 0 && kind < kNumKinds) ? kKindNames[kind] : nullptr;
}

int moe_profile_read(double* total_ms, uint64_t* launches, int n) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (const ProfRec& r : g_prof_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      g_prof_ms[r.kind] += ms;
      g_prof_n[r.kind] += 1;
    }
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_prof_pending.clear();
  for (int i = 0; i < kNumKinds && i < n; ++i) {
    if (total_ms) total_ms[i] = g_prof_ms[i];
    if (launches) launches[i] = g_prof_n[i];
  }
  for (int i = 0; i < kNumKinds; ++i) {
    g_prof_ms[i] = 0.0;
    g_prof_n[i] = 0;
  }
  return kNumKinds;
}

const char* moe_status_string(moe_status st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported (needs an sm_103 GPU and a supported shape)";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_BAD_INDEX: return "expert index out of range";
    case MOE_ERR_TIMEOUT: return "device pipeline wait timed out";
    case MOE_ERR_CUDA: return "CUDA call failed";
  }
  return "unknown status";
}

moe_status moe_get_device_error(void* ws, moe_stream_t stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  MOE_CUDA(cudaStreamSynchronize(st));
  int code = 0;
  MOE_CUDA(cudaMemcpy(&code, ws, sizeof(int), cudaMemcpyDeviceToHost));
  if (code != 0) MOE_CUDA(cudaMemset(ws, 0, sizeof(int)));
  return static_cast<moe_status>(code);
}

moe_status moe_plan(const moe_shape* s, const int32_t* topk_idx, const moe_plan_t* plan, void* ws,
                    size_t ws_bytes, moe_stream_t stream) {
  if (!shape_ok(s) || !plan || !ws || !plan->counts || !plan->offsets) return MOE_ERR_INVALID_ARG;
  const int64_t Tk = s->T * s->k;
  if (Tk > 0 && (!topk_idx || !plan->perm || !plan->inv)) return MOE_ERR_INVALID_ARG;
  const Layout L = layout(s, 0);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  int sms = 0;
  const moe_status ds = device_info(&sms);
  if (ds != MOE_OK) return ds;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  MOE_CUDA(tracked(kKPlan, Tk > 0 ? 3 : 1, st, [&] {
    return launch_plan(topk_idx, Tk, s->E, plan->counts, plan->offsets, plan->perm, plan->inv,
                       at<int>(ws, L.poff), at<int>(ws, L.blkhist), at<int>(ws, L.err), st);
  }));
  return MOE_OK;
}

moe_status moe_route(const moe_shape* s, const float* logits, int32_t* topk_idx, float* topk_w,
                     const moe_plan_t* plan, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!shape_ok(s)) return MOE_ERR_INVALID_ARG;
  if (plan && (!ws || !plan->counts || !plan->offsets)) return MOE_ERR_INVALID_ARG;
  const int64_t Tk = s->T * s->k;
  if (s->T > 0 && (!logits || !topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
  if (plan && Tk > 0 && (!plan->perm || !plan->inv)) return MOE_ERR_INVALID_ARG;
  if (plan && ws_bytes < layout(s, 0).total) return MOE_ERR_WORKSPACE;
  int sms = 0;
  const moe_status ds = device_info(&sms);
  if (ds != MOE_OK) return ds;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (s->T > 0) {
    MOE_CUDA(tracked(kKRoute, 1, st, [&] {
      return launch_route(logits, s->T, s->E, s->k, topk_idx, topk_w, sms, st);
    }));
  }
  if (!plan) return MOE_OK;
  return moe_plan(s, topk_idx, plan, ws, ws_bytes, stream);
}

moe_status moe_ffn_fwd(const moe_shape* s, const void* x, const int32_t* topk_idx,
                       const float* topk_w, const void* w_gate_up, const void* w_down,
                       const moe_bias_t* bias_in, const moe_plan_t* plan, void* y, void* saved,
                       void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!shape_ok(s) || !ws || !w_gate_up || !w_down) return MOE_ERR_INVALID_ARG;
  const moe_bias_t bias = bias_or_none(bias_in);
  if (!bias_aligned(bias)) return MOE_ERR_INVALID_ARG;
  if (s->T == 0) return MOE_OK;
  if (!x || !topk_idx || !topk_w || !y) return MOE_ERR_INVALID_ARG;
  if (plan && (!plan->counts || !plan->offsets || !plan->perm || !plan->inv))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(w_gate_up) || !aligned16(w_down) ||
      (saved && !aligned16(saved)))
    return MOE_ERR_INVALID_ARG;
  const Layout L = layout(s, 1);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  int sms = 0;
  const moe_status ds = device_info(&sms);
  if (ds != MOE_OK) return ds;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  const int es = elem_bytes(s);
  const int64_t Tk = s->T * s->k;
  const int64_t R = rows_max(s);
  const int H = s->H, I = s->I, E = s->E;
  int* err = at<int>(ws, L.err);
  int* poff = at<int>(ws, L.poff);
  const int *counts, *offsets, *perm, *inv;
  if (plan) {
    counts = plan->counts;
    offsets = plan->offsets;
    perm = plan->perm;
    inv = plan->inv;
    MOE_CUDA(tracked(kKOffsets, 1, st, [&] { return launch_padded_offsets(counts, E, poff, st); }));
  } else {
    int* c = at<int>(ws, L.counts);
    int* o = at<int>(ws, L.offsets);
    int* p = at<int>(ws, L.perm);
    int* v = at<int>(ws, L.inv);
    MOE_CUDA(tracked(kKPlan, 3, st, [&] {
      return launch_plan(topk_idx, Tk, E, c, o, p, v, poff, at<int>(ws, L.blkhist), err, st);
    }));
    counts = c;
    offsets = o;
    perm = p;
    inv = v;
  }
  // the training forward gathers straight into the saved context, which the
  // backward reads instead of gathering x again
  void* xp = saved ? saved : at<char>(ws, L.xp);
  void* aact = at<char>(ws, L.act);
  void* h1_saved = saved ? static_cast<void*>(static_cast<char*>(saved) + saved_h1_offset(s))
                         : nullptr;
  MOE_CUDA(tracked(kKGather, 1, st, [&] {
    return launch_gather_rows(x, H, s->k, E, poff, counts, offsets, perm, static_cast<int>(Tk),
                              R, xp, es, sms, st);
  }));

  const moe_status gs = enqueue_gate_up(s, xp, w_gate_up, bias.b_gate_up,
                                        es == 4 ? at<float>(ws, L.wguT) : nullptr, aact, h1_saved,
                                        poff, counts, offsets, perm, topk_w, err, sms, st);
  if (gs != MOE_OK) return gs;

  const uint32_t BK = 128 / es, CH = 128 / es;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  const uint32_t AROWS = 128;

  // down GEMM * routing weight -> fp32 rows Ow
  float* ow = at<float>(ws, L.ow);
  GemmMaps m2;
  bool ok = map2d(&m2.a, es, aact, I, R, I, BK, AROWS, SW);
  if (es == 2) {
    ok = ok && map3d(&m2.b0, es, w_down, H, I, E, H, static_cast<int64_t>(H) * I, CH, BK, SW);
  } else {
    float* wdT = at<float>(ws, L.wdT);
    MOE_CUDA(tracked(kKTranspose, 1, st, [&] {
      return launch_transpose_f32(static_cast<const float*>(w_down), wdT, E, I, H, st);
    }));
    ok = ok && map3d(&m2.b0, es, wdT, I, H, E, I, static_cast<int64_t>(H) * I, BK, 256, SW);
  }
  if (!ok) return MOE_ERR_CUDA;
  // bf16 tiles tokens on the MMA's N side; short units use a 32-row box
  m2.a2 = m2.a;
  if (es == 2 && !map2d(&m2.a2, es, aact, I, R, I, BK, 32, SW)) return MOE_ERR_CUDA;
  m2.b1 = m2.b0;
  GemmArgs a2 = base_args(s, poff, counts, offsets, perm, topk_w, err);
  a2.out[0] = out_view(ow, H, R, H);
  a2.bias = bias.b_down;
  a2.num_kb = (I + BK - 1) / BK;
  a2.n_tiles = (H + gemm_block_n(kFwdDown, es) - 1) / gemm_block_n(kFwdDown, es);
  MOE_CUDA(tracked(kKFwdDown, 1, st, [&] { return launch_gemm(kFwdDown, es, m2, a2, sms, st); }));

  // combine (y in the storage dtype, or fp32 on request)
  const int y_bytes = s->out_fp32 ? 4 : es;
  MOE_CUDA(tracked(kKCombine, 1, st, [&] {
    return launch_combine(ow, H, s->k, E, topk_idx, inv, offsets, poff, s->T, R, y, y_bytes, sms,
                          st);
  }));
  return MOE_OK;
}

moe_status moe_ffn_bwd(const moe_shape* s, const void* dy, const void* x, const int32_t* topk_idx,
                       const float* topk_w, const void* w_gate_up, const void* w_down,
                       const moe_bias_t* bias_in, const moe_plan_t* plan, const void* saved,
                       void* dx, float* d_topk_w, float* dw_gate_up, float* dw_down, void* ws,
                       size_t ws_bytes, moe_stream_t stream) {
  if (!shape_ok(s) || !ws || !w_gate_up || !w_down || !dw_gate_up || !dw_down)
    return MOE_ERR_INVALID_ARG;
  const moe_bias_t bias = bias_or_none(bias_in);
  if (!bias_aligned(bias)) return MOE_ERR_INVALID_ARG;
  int sms = 0;
  const moe_status ds = device_info(&sms);
  if (ds != MOE_OK) return ds;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int es = elem_bytes(s);
  const int H = s->H, I = s->I, E = s->E;
  if (s->T == 0) {
    MOE_CUDA(tracked(kKMemset, 2, st, [&] {
      cudaError_t e1 = cudaMemsetAsync(dw_gate_up, 0, sizeof(float) * E * H * 2ull * I, st);
      cudaError_t e2 = cudaMemsetAsync(dw_down, 0, sizeof(float) * E * static_cast<size_t>(I) * H, st);
      return e1 != cudaSuccess ? e1 : e2;
    }));
    if (bias.db_gate_up)
      MOE_CUDA(tracked(kKMemset, 1, st, [&] {
        return cudaMemsetAsync(bias.db_gate_up, 0, sizeof(float) * E * 2ull * I, st);
      }));
    if (bias.db_down)
      MOE_CUDA(tracked(kKMemset, 1, st, [&] {
        return cudaMemsetAsync(bias.db_down, 0, sizeof(float) * E * static_cast<size_t>(H), st);
      }));
    return MOE_OK;
  }
  if (!dy || !x || !topk_idx || !topk_w || !plan || !dx || !d_topk_w)
    return MOE_ERR_INVALID_ARG;
  if (!plan->counts || !plan->offsets || !plan->perm || !plan->inv) return MOE_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(x) || !aligned16(dx) || (saved && !aligned16(saved)) ||
      !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(dw_gate_up) ||
      !aligned16(dw_down))
    return MOE_ERR_INVALID_ARG;
  // without a saved context the backward recomputes it (workspace kind 3)
  const bool recompute = (saved == nullptr);
  const Layout L = layout(s, recompute ? 3 : 2);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;

  const int64_t Tk = s->T * s->k;
  const int64_t R = rows_max(s);
  int* err = at<int>(ws, L.err);
  int* poff = at<int>(ws, L.poff);
  const int* counts = plan->counts;
  const int* offsets = plan->offsets;
  const int* perm = plan->perm;
  const int* inv = plan->inv;
  MOE_CUDA(tracked(kKOffsets, 1, st, [&] { return launch_padded_offsets(counts, E, poff, st); }));
  // bf16: which experts' weight gradients need the bf16 remainder parts
  const int* lo_flags = nullptr;
  if (es == 2) {
    int* f = at<int>(ws, L.lo_flags);
    MOE_CUDA(tracked(kKSplitSelect, 1, st, [&] {
      return launch_split_select(offsets, perm, topk_w, static_cast<int>(Tk), E, kSplitMinNeff, f,
                                 st);
    }));
    lo_flags = f;
  }

  void* dyp = at<char>(ws, L.dyp);
  // the forward's expert-grouped x rows and pre-activations: saved, or
  // recomputed here by the forward's gather and gate_up GEMM (bit-identical)
  void* xp = recompute ? at<char>(ws, L.xp) : const_cast<void*>(saved);
  const void* h1_saved =
      recompute ? static_cast<const void*>(at<char>(ws, L.h1))
                : static_cast<const void*>(static_cast<const char*>(saved) +
                                           saved_h1_offset(s));
  void* dh1 = at<char>(ws, L.dh1);
  void* aw = at<char>(ws, L.aw);
  const bool split = (es == 2);
  void* dh1lo = split ? at<char>(ws, L.dh1lo) : dh1;
  void* awlo = split ? at<char>(ws, L.awlo) : aw;
  float* dwpart = at<float>(ws, L.dwpart);
  MOE_CUDA(tracked(kKGather, 1, st, [&] {
    return launch_gather_rows(dy, H, s->k, E, poff, counts, offsets, perm, static_cast<int>(Tk),
                              R, dyp, es, sms, st);
  }));
  if (recompute) {
    MOE_CUDA(tracked(kKGather, 1, st, [&] {
      return launch_gather_rows(x, H, s->k, E, poff, counts, offsets, perm, static_cast<int>(Tk),
                                R, xp, es, sms, st);
    }));
    // the activation output is not needed: it goes to the dH1 region, which
    // the down dgrad overwrites
    const moe_status gs =
        enqueue_gate_up(s, xp, w_gate_up, bias.b_gate_up, es == 4 ? at<float>(ws, L.wguT) : nullptr,
                        dh1, const_cast<void*>(h1_saved), poff, counts, offsets, perm, topk_w,
                        err, sms, st);
    if (gs != MOE_OK) return gs;
  }

  const uint32_t BK = 128 / es, CH = 128 / es;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  const size_t up_off = static_cast<size_t>(I) * es;
  bool ok;

  // TF32 reads only the top bits of fp32 operands: give the dgrads
  // round-to-nearest copies of the weights.
  const void* wd_op = w_down;
  const void* wgu_op = w_gate_up;
  if (!split) {
    float* wdR = at<float>(ws, L.wdR);
    float* wguR = at<float>(ws, L.wguR);
    MOE_CUDA(tracked(kKTranspose, 2, st, [&] {
      cudaError_t e1 = launch_round_copy_tf32(static_cast<const float*>(w_down), wdR,
                                              static_cast<int64_t>(E) * I * H, sms, st);
      cudaError_t e2 = launch_round_copy_tf32(static_cast<const float*>(w_gate_up), wguR,
                                              static_cast<int64_t>(E) * 2 * I * H, sms, st);
      return e1 != cudaSuccess ? e1 : e2;
    }));
    wd_op = wdR;
    wgu_op = wguR;
  }

  // (1) down dgrad + activation backward -> dH1 (gate | up), w*a, dw partials
  GemmMaps m1;
  const uint32_t AROWS = 128;
  ok = map2d(&m1.a, es, dyp, H, R, H, BK, AROWS, SW) &&
       map3d(&m1.b0, es, wd_op, H, I, E, H, static_cast<int64_t>(H) * I, BK,
             dgrad_b_rows(kDgradDown, es), SW);
  if (!ok) return MOE_ERR_CUDA;
  m1.a2 = m1.a;
  m1.b1 = m1.b0;
  GemmArgs a1 = base_args(s, poff, counts, offsets, perm, topk_w, err);
  a1.num_kb = (H + BK - 1) / BK;
  a1.n_tiles = dgrad_down_ntiles(s);
  a1.h1 = h1_saved;
  a1.dwpart = dwpart;
  a1.lo_flags = lo_flags;
  // interleaved gate_up columns: dgate / dup pairs over all 2I columns
  const bool il = s->gate_up_layout == MOE_GATE_UP_INTERLEAVED;
  a1.out[0] = out_view(dh1, 2ll * I, R, il ? 2ll * I : I);
  a1.out[1] = out_view(static_cast<char*>(dh1) + up_off, 2ll * I, R, I);
  a1.out[2] = out_view(aw, I, R, I);
  a1.out[3] = out_view(dh1lo, 2ll * I, R, il ? 2ll * I : I);
  a1.out[4] = out_view(static_cast<char*>(dh1lo) + up_off, 2ll * I, R, I);
  a1.out[5] = out_view(awlo, I, R, I);
  MOE_CUDA(tracked(kKDgradDown, 1, st, [&] { return launch_gemm(kDgradDown, es, m1, a1, sms, st); }));
  // with a down bias, o = a Wd + b_down, so d(topk w) gains <dY, b_down>: one
  // more partial row, summed last
  if (bias.b_down)
    MOE_CUDA(tracked(kKBiasDot, 1, st, [&] {
      return launch_bias_slot_dot(dy, bias.b_down, H, s->k, E, topk_idx, inv, offsets, poff, Tk,
                                  R, dwpart + static_cast<int64_t>(a1.n_tiles) * R, es, sms, st);
    }));
  MOE_CUDA(tracked(kKDwReduce, 1, st, [&] {
    return launch_dw_reduce(dwpart, a1.n_tiles + (bias.b_down ? 1 : 0), R, E, topk_idx, inv,
                            offsets, poff, Tk, d_topk_w, st);
  }));
  // bias gradients: per-expert column sums of dH1 (hi + lo) and of w * dy
  // (dy read in token order through the plan)
  if (bias.db_gate_up)
    MOE_CUDA(tracked(kKBiasGrad, 1, st, [&] {
      return launch_expert_colsum(dh1, split ? dh1lo : nullptr, 2 * I, 2ll * I, 0, E, poff,
                                  counts, offsets, perm, topk_w, static_cast<int>(Tk), false,
                                  lo_flags, bias.db_gate_up, es, st);
    }));
  if (bias.db_down)
    MOE_CUDA(tracked(kKBiasGrad, 1, st, [&] {
      return launch_expert_colsum(dy, nullptr, H, H, s->k, E, poff, counts, offsets, perm,
                                  topk_w, static_cast<int>(Tk), true, nullptr, bias.db_down, es,
                                  st);
    }));

  // (2) down wgrad: dWd[e] = (w*a)_e^T dYp_e  (w*a as a bf16 hi/lo pair)
  GemmMaps m2;
  ok = true;
  if (split) {
    ok = map2d(&m2.a, es, aw, I, R, I, CH, BK, SW) &&
         map2d(&m2.a2, es, awlo, I, R, I, CH, BK, SW) && map2d(&m2.b0, es, dyp, H, R, H, CH, BK, SW);
  } else {
    // TF32: K-major copies [I, R] and [H, R] of the row-major activations
    float* awT = at<float>(ws, L.awT);
    float* dypT = at<float>(ws, L.dypT);
    MOE_CUDA(tracked(kKTranspose, 2, st, [&] {
      cudaError_t e1 = launch_transpose_f32(static_cast<const float*>(aw), awT, 1, R, I, st);
      cudaError_t e2 = launch_transpose_f32(static_cast<const float*>(dyp), dypT, 1, R, H, st);
      return e1 != cudaSuccess ? e1 : e2;
    }));
    ok = ok && map2d(&m2.a, es, awT, R, I, R, BK, 128, SW) &&
         map2d(&m2.b0, es, dypT, R, H, R, BK, 256, SW);
    m2.a2 = m2.a;
  }
  if (!ok) return MOE_ERR_CUDA;
  m2.b1 = m2.b0;
  GemmArgs a2 = base_args(s, poff, counts, offsets, perm, topk_w, err);
  a2.lo_flags = lo_flags;
  a2.out[0] = out_view(dw_down, H, I, H, static_cast<int64_t>(I) * H);
  if (!map3d(&m2.out, 4, dw_down, H, I, E, H, static_cast<int64_t>(I) * H, 32, 32, SW))
    return MOE_ERR_CUDA;
  a2.m_tiles = (I + 127) / 128;
  a2.n_tiles = (H + gemm_block_n(kWgradDown, es) - 1) / gemm_block_n(kWgradDown, es);
  MOE_CUDA(tracked(kKWgradDown, 1, st, [&] { return launch_gemm(kWgradDown, es, m2, a2, sms, st); }));

  // (3) gate_up dgrad: dXp = dH1 Wgu[e]^T  (fp32 rows for the combine)
  float* dxp = at<float>(ws, L.dxp);
  GemmMaps m3;
  ok = map2d(&m3.a, es, dh1, 2ll * I, R, 2ll * I, BK, AROWS, SW) &&
       map3d(&m3.b0, es, wgu_op, 2ll * I, H, E, 2ll * I, 2ll * I * H, BK,
             dgrad_b_rows(kDgradGateUp, es), SW);
  if (!ok) return MOE_ERR_CUDA;
  m3.a2 = m3.a;
  if (split && !map2d(&m3.a2, es, dh1, 2ll * I, R, 2ll * I, BK, 32, SW)) return MOE_ERR_CUDA;
  m3.b1 = m3.b0;
  GemmArgs a3 = base_args(s, poff, counts, offsets, perm, topk_w, err);
  a3.out[0] = out_view(dxp, H, R, H);
  a3.num_kb = (2 * I + BK - 1) / BK;
  a3.n_tiles = (H + gemm_block_n(kDgradGateUp, es) - 1) / gemm_block_n(kDgradGateUp, es);
  MOE_CUDA(tracked(kKDgradGateUp, 1, st, [&] { return launch_gemm(kDgradGateUp, es, m3, a3, sms, st); }));
  MOE_CUDA(tracked(kKCombine, 1, st, [&] {
    return launch_combine(dxp, H, s->k, E, topk_idx, inv, offsets, poff, s->T, R, dx,
                          s->out_fp32 ? 4 : es, sms, st);
  }));

  // (4) gate_up wgrad: dWgu[e] = Xp_e^T dH1_e  (dH1 as a bf16 hi/lo pair)
  const int bn4 = gemm_block_n(kWgradGateUp, es);
  GemmMaps m4;
  ok = true;
  if (split) {
    ok = map2d(&m4.a, es, xp, H, R, H, CH, BK, SW) &&
         map2d(&m4.b0, es, dh1, 2ll * I, R, 2ll * I, CH, BK, SW) &&
         map2d(&m4.b1, es, dh1lo, 2ll * I, R, 2ll * I, CH, BK, SW);
  } else {
    float* xpT = at<float>(ws, L.xpT);
    float* dh1T = at<float>(ws, L.dh1T);
    MOE_CUDA(tracked(kKTranspose, 2, st, [&] {
      cudaError_t e1 = launch_transpose_f32(static_cast<const float*>(xp), xpT, 1, R, H, st);
      cudaError_t e2 = launch_transpose_f32(static_cast<const float*>(dh1), dh1T, 1, R, 2 * I, st);
      return e1 != cudaSuccess ? e1 : e2;
    }));
    ok = ok && map2d(&m4.a, es, xpT, R, H, R, BK, 128, SW) &&
         map2d(&m4.b0, es, dh1T, R, 2ll * I, R, BK, 256, SW);
    m4.b1 = m4.b0;
  }
  if (!ok) return MOE_ERR_CUDA;
  m4.a2 = m4.a;
  GemmArgs a4 = base_args(s, poff, counts, offsets, perm, topk_w, err);
  a4.lo_flags = lo_flags;
  a4.out[0] = out_view(dw_gate_up, 2ll * I, H, 2ll * I, 2ll * I * H);
  if (!map3d(&m4.out, 4, dw_gate_up, 2ll * I, H, E, 2ll * I, 2ll * I * H, 32, 32, SW))
    return MOE_ERR_CUDA;
  a4.m_tiles = (H + gemm_block_m(kWgradGateUp, es) - 1) / gemm_block_m(kWgradGateUp, es);
  a4.n_tiles = (2 * I + bn4 - 1) / bn4;
  MOE_CUDA(tracked(kKWgradGateUp, 1, st, [&] { return launch_gemm(kWgradGateUp, es, m4, a4, sms, st); }));
  return MOE_OK;
}

moe_status moe_gather_rows(const int32_t* index, int64_t n, int32_t div, const void* src,
                           int64_t src_rows, int64_t row_bytes, void* dst, moe_stream_t stream) {
  if (n < 0 || div < 1 || row_bytes <= 0 || (row_bytes % 4) || src_rows < 0 ||
      row_bytes / 4 > (1ll << 30))
    return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (!index || !dst || (!src && src_rows > 0)) return MOE_ERR_INVALID_ARG;
  int sms = 0;
  const moe_status ds = device_info(&sms);
  if (ds != MOE_OK) return ds;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  MOE_CUDA(tracked(kKGatherIndex, 1, st, [&] {
    return launch_gather_index(index, n, div, src, src_rows, row_bytes, dst, sms, st);
  }));
  return MOE_OK;
}

moe_status moe_combine_rows(const moe_shape* s, const int32_t* inv, const float* topk_w,
                            const void* src, int32_t src_fp32, void* dst, moe_stream_t stream) {
  if (!shape_ok(s) || (src_fp32 != 0 && src_fp32 != 1)) return MOE_ERR_INVALID_ARG;
  if (s->T == 0) return MOE_OK;
  if (!inv || !src || !dst || !aligned16(src) || !aligned16(dst)) return MOE_ERR_INVALID_ARG;
  int sms = 0;
  const moe_status ds = device_info(&sms);
  if (ds != MOE_OK) return ds;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int es = elem_bytes(s);
  MOE_CUDA(tracked(kKCombineDense, 1, st, [&] {
    return launch_combine_dense(src, src_fp32 ? 4 : es, s->H, s->k, inv, topk_w, s->T, dst,
                                s->out_fp32 ? 4 : es, sms, st);
  }));
  return MOE_OK;
}

}  // extern "C"
