// Row movement between token order and the tile-padded expert-grouped order:
//   gather   ("sparse token extraction" / "each token is repeated k times")
//   combine  (the accumulate-back step the dispatch-and-combine page does with
//             index_add_; here a k-way gather-sum per token in a fixed order,
//             so no float atomics and bitwise-reproducible results; its
//             inputs are the fp32 rows the GEMM epilogues write)
//   dw_reduce (fixed-order sum of the per-column-tile partial dot products
//             that make d(topk weights))
//   bias terms (the optional per-expert biases: the b_down term of
//             d(topk weights) and the per-expert column sums that are the
//             bias gradients)
// All are HBM-bound and use 16-byte vector accesses.  The row kernels run one
// warp per row on a grid sized as a multiple of the SM count; the column sums
// run one thread per 8 columns of one expert.
#include <algorithm>

#include "kernels.h"

namespace moe {

// Expert whose padded segment holds row p: largest e with poff[e] <= p.
__device__ __forceinline__ int expert_of_row(const int* __restrict__ poff, int E, int p) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(poff + mid) <= p)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Row of slot s in the padded layout, or -1 when the slot's expert id is out
// of range or the row falls outside the expert's live rows (an inconsistent
// plan): such slots contribute nothing instead of reading out of bounds.
__device__ __forceinline__ int64_t padded_row_of_slot(int s, int E, const int* __restrict__ idx,
                                                      const int* __restrict__ inv,
                                                      const int* __restrict__ offsets,
                                                      const int* __restrict__ poff) {
  const int e = __ldg(idx + s);
  if (e < 0 || e >= E) return -1;
  const int local = __ldg(inv + s) - __ldg(offsets + e);
  if (local < 0 || local >= __ldg(offsets + e + 1) - __ldg(offsets + e)) return -1;
  return static_cast<int64_t>(__ldg(poff + e)) + local;
}

__global__ void __launch_bounds__(256) gather_rows_kernel(
    const uint4* __restrict__ src, int vec_per_row, int k, int E, const int* __restrict__ poff,
    const int* __restrict__ counts, const int* __restrict__ offsets, const int* __restrict__ perm,
    int tk, int64_t rows_max, int tf32, uint4* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  // never past the workspace bound, even for an inconsistent caller plan
  const int64_t rows = min(static_cast<int64_t>(__ldg(poff + E)), rows_max);
  for (int64_t p = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       p < rows; p += warps) {
    const int e = expert_of_row(poff, E, static_cast<int>(p));
    const int local = static_cast<int>(p) - __ldg(poff + e);
    uint4* d = dst + p * vec_per_row;
    const int gi = __ldg(offsets + e) + local;
    const int slot = (local < __ldg(counts + e) && gi < tk) ? __ldg(perm + gi) : -1;
    if (slot >= 0 && slot < tk) {
      const uint4* sr = src + static_cast<int64_t>(slot / k) * vec_per_row;
      if (tf32) {
        for (int v = lane; v < vec_per_row; v += 32) {
          const uint4 a = __ldg(sr + v);
          d[v] = make_uint4(__float_as_uint(round_tf32(__uint_as_float(a.x))),
                            __float_as_uint(round_tf32(__uint_as_float(a.y))),
                            __float_as_uint(round_tf32(__uint_as_float(a.z))),
                            __float_as_uint(round_tf32(__uint_as_float(a.w))));
        }
      } else {
        for (int v = lane; v < vec_per_row; v += 32) d[v] = __ldg(sr + v);
      }
    } else {
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int v = lane; v < vec_per_row; v += 32) d[v] = z;
    }
  }
}

constexpr int kMaxK = 32;

__device__ __forceinline__ void store8(__nv_bfloat16* out, const float* a) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
  *reinterpret_cast<uint4*>(out) = v;
}
__device__ __forceinline__ void store8(float* out, const float* a) {
  reinterpret_cast<float4*>(out)[0] = make_float4(a[0], a[1], a[2], a[3]);
  reinterpret_cast<float4*>(out)[1] = make_float4(a[4], a[5], a[6], a[7]);
}

// src: fp32 rows of the padded layout [rows_max, H]; out: [T, H] of OutT.
// One warp per token, 8 columns per lane per step.
template <typename OutT>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ src, int H, int k,
                                                      int E, const int* __restrict__ idx,
                                                      const int* __restrict__ inv,
                                                      const int* __restrict__ offsets,
                                                      const int* __restrict__ poff, int64_t T_,
                                                      int64_t rows_max, OutT* __restrict__ out) {
  __shared__ int64_t rows_s[8][kMaxK];   // padded rows of the current token's k slots
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int groups = H / 8;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + wib; t < T_;
       t += warps) {
    if (lane < k)
      rows_s[wib][lane] =
          padded_row_of_slot(static_cast<int>(t * k + lane), E, idx, inv, offsets, poff);
    __syncwarp();
    for (int v = lane; v < groups; v += 32) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      for (int j = 0; j < k; ++j) {
        const int64_t r = rows_s[wib][j];
        if (r >= 0 && r < rows_max) {
          const float4* p = reinterpret_cast<const float4*>(src + r * H + v * 8);
          const float4 a = __ldg(p), b = __ldg(p + 1);
          acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
          acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
        }
      }
      store8(out + t * H + v * 8, acc);
    }
    __syncwarp();
  }
}

// out[b][c][r] = tf32_round(in[b][r][c]) (fp32), 32x32 tiles through shared
// memory: K-major TF32 operands for the fp32 path.
__global__ void __launch_bounds__(256) transpose_f32_kernel(const float* __restrict__ in,
                                                            float* __restrict__ out, int rows,
                                                            int cols) {
  __shared__ float tile[32][33];
  const int64_t plane = static_cast<int64_t>(rows) * cols;
  in += blockIdx.z * plane;
  out += blockIdx.z * plane;
  const int c0 = blockIdx.x * 32;
  for (int r0 = blockIdx.y * 32; r0 < rows; r0 += gridDim.y * 32) {
    for (int i = threadIdx.y; i < 32; i += 8) {
      const int r = r0 + i, c = c0 + threadIdx.x;
      if (r < rows && c < cols) tile[i][threadIdx.x] = in[static_cast<int64_t>(r) * cols + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += 8) {
      const int c = c0 + i, r = r0 + threadIdx.x;
      if (r < rows && c < cols)
        out[static_cast<int64_t>(c) * rows + r] = round_tf32(tile[threadIdx.x][i]);
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(256) dw_reduce_kernel(const float* __restrict__ dwpart,
                                                        int ntiles, int64_t rows_max, int E,
                                                        const int* __restrict__ idx,
                                                        const int* __restrict__ inv,
                                                        const int* __restrict__ offsets,
                                                        const int* __restrict__ poff, int64_t Tk,
                                                        float* __restrict__ d_topk_w) {
  const int64_t s = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (s >= Tk) return;
  const int64_t p = padded_row_of_slot(static_cast<int>(s), E, idx, inv, offsets, poff);
  float acc = 0.f;
  if (p >= 0 && p < rows_max)
    for (int n = 0; n < ntiles; ++n) acc += __ldg(dwpart + n * rows_max + p);
  d_topk_w[s] = acc;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* a) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    a[2 * i] = f.x;
    a[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float* a) {
  const float4 x = __ldg(reinterpret_cast<const float4*>(p));
  const float4 y = __ldg(reinterpret_cast<const float4*>(p) + 1);
  a[0] = x.x; a[1] = x.y; a[2] = x.z; a[3] = x.w;
  a[4] = y.x; a[5] = y.y; a[6] = y.z; a[7] = y.w;
}

// Bias term of d(topk weights): <dy[t], b_down[e]> for each slot s = t*k + j
// routed to expert e, written at the slot's padded row.  One warp per slot;
// it reads dy in token order (the k slots of a token run on neighbouring
// warps, so a token's row comes from HBM once) and the bias row from L2.
template <typename T>
__global__ void __launch_bounds__(256) bias_slot_dot_kernel(
    const T* __restrict__ dy, const T* __restrict__ bd, int H, int k, int E,
    const int* __restrict__ idx, const int* __restrict__ inv, const int* __restrict__ offsets,
    const int* __restrict__ poff, int64_t Tk, int64_t rows_max, float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t s = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       s < Tk; s += warps) {
    const int64_t p = padded_row_of_slot(static_cast<int>(s), E, idx, inv, offsets, poff);
    if (p < 0 || p >= rows_max) continue;
    const T* dr = dy + (s / k) * H;
    const T* br = bd + static_cast<int64_t>(__ldg(idx + s)) * H;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int c = lane * 8;
    for (; c + 3 * 256 < H; c += 4 * 256) {   // four 16-byte loads of each in flight
      float a[4][8], b[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        load8(dr + c + u * 256, a[u]);
        load8(br + c + u * 256, b[u]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[u] = fmaf(a[u][i], b[u][i], acc[u]);
    }
    for (; c < H; c += 256) {
      float a[8], b[8];
      load8(dr + c, a);
      load8(br + c, b);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[0] = fmaf(a[i], b[i], acc[0]);
    }
    float v = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    if (lane == 0) out[p] = v;
  }
}

// Per-expert column sums over the expert's rows j = 0 .. counts[e]-1: the
// bias gradients (dH1, its bf16 hi and lo parts added back together, for
// b_gate_up; w * dy for b_down).  Row j is row poff[e] + j of src, or, with
// gather_k > 0, token row perm[offsets[e] + j] / gather_k (dy in token order,
// which stays in L2 while the expert rows are read).  A block takes 512
// columns of one expert (blockIdx.y): 64 threads x 8 columns, and kRowGroups
// groups of them take every kRowGroups-th row; the groups' sums are added in
// group order at the end, so the result does not depend on timing.
constexpr int kRowGroups = 4;

template <typename T>
__global__ void __launch_bounds__(64 * kRowGroups) expert_colsum_kernel(
    const T* __restrict__ src, const T* __restrict__ src2, int C, int64_t ld, int gather_k,
    const int* __restrict__ poff, const int* __restrict__ counts,
    const int* __restrict__ offsets, const int* __restrict__ perm,
    const float* __restrict__ topk_w, int tk, int weighted, const int* __restrict__ src2_flags,
    float* __restrict__ out) {
  __shared__ float4 part[kRowGroups][64][2];
  const int e = blockIdx.y;
  // src2 (a bf16 remainder) exists only for experts whose flag is set
  if (src2_flags && __ldg(src2_flags + e) == 0) src2 = nullptr;
  const int tx = threadIdx.x, g = threadIdx.y;
  const int c = (blockIdx.x * 64 + tx) * 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  if (c < C) {
    const int p0 = __ldg(poff + e);
    const int n = min(__ldg(counts + e), __ldg(poff + e + 1) - p0);
    const int g0 = __ldg(offsets + e);
    const bool need_slot = gather_k > 0 || weighted;
#pragma unroll 4
    for (int j = g; j < n; j += kRowGroups) {
      int slot = 0;
      if (need_slot) {
        const int gi = g0 + j;
        slot = gi < tk ? __ldg(perm + gi) : -1;
        if (slot < 0 || slot >= tk) continue;   // an inconsistent plan: contributes nothing
      }
      const int64_t r =
          (gather_k > 0 ? static_cast<int64_t>(slot / gather_k) : static_cast<int64_t>(p0 + j)) *
              ld + c;
      float a[8];
      load8(src + r, a);
      if (src2) {
        float b[8];
        load8(src2 + r, b);
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] += b[i];
      }
      const float sc = weighted ? __ldg(topk_w + slot) : 1.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(sc, a[i], acc[i]);
    }
  }
  part[g][tx][0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  part[g][tx][1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  __syncthreads();
  if (g == 0 && c < C) {
#pragma unroll
    for (int q = 1; q < kRowGroups; ++q) {
      const float4 x = part[q][tx][0], y = part[q][tx][1];
      acc[0] += x.x; acc[1] += x.y; acc[2] += x.z; acc[3] += x.w;
      acc[4] += y.x; acc[5] += y.y; acc[6] += y.z; acc[7] += y.w;
    }
    store8(out + static_cast<int64_t>(e) * C + c, acc);
  }
}

// Whether each expert's weight gradients need the bf16 remainder (lo) part of
// their computed operand (dH1 for gate_up, w*a for down).  Without it the
// operand is rounded to bf16 once, a relative error of up to 2^-8 per value.
// In a weight-gradient element, a sum over the expert's rows, those errors
// average out unless a few rows dominate the sum; the routing weight scales
// every row, so the number of rows that count is the effective row count
// n_eff = (sum w^2)^2 / sum w^4 over the expert's rows (n_eff = n for equal
// weights).  Experts with n_eff >= min_neff get flag 0 (one bf16 operand);
// the rest, and experts without rows, flag 1 (hi + lo).  One warp per
// expert, fixed summation order.
__global__ void __launch_bounds__(256) split_select_kernel(
    const int* __restrict__ offsets, const int* __restrict__ perm,
    const float* __restrict__ topk_w, int tk, int E, float min_neff, int* __restrict__ lo_flags) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (e >= E) return;
  const int g0 = __ldg(offsets + e), g1 = min(__ldg(offsets + e + 1), tk);
  float s2 = 0.f, s4 = 0.f;
  for (int gi = g0 + lane; gi < g1; gi += 32) {
    const int slot = __ldg(perm + gi);
    const float w = (slot >= 0 && slot < tk) ? __ldg(topk_w + slot) : 0.f;
    const float w2 = w * w;
    s2 += w2;
    s4 = fmaf(w2, w2, s4);
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    s2 += __shfl_xor_sync(0xffffffffu, s2, d);
    s4 += __shfl_xor_sync(0xffffffffu, s4, d);
  }
  // (all-zero weights make the operand exactly zero: no remainder needed;
  // non-finite weights fail the comparison and keep the remainder)
  if (lane == 0) lo_flags[e] = (g1 > g0 && s2 * s2 >= min_neff * s4) ? 0 : 1;
}

cudaError_t launch_split_select(const int* offsets, const int* perm, const float* topk_w, int tk,
                                int E, float min_neff, int* lo_flags, cudaStream_t st) {
  split_select_kernel<<<(E + 7) / 8, 256, 0, st>>>(offsets, perm, topk_w, tk, E, min_neff,
                                                   lo_flags);
  return cudaGetLastError();
}

// ---- dense row movement for the expert-parallel exchange ----------------
// dst[r] = src[index[r] / div] for r < n, rows of row_bytes bytes (a multiple
// of 4; 16-byte accesses when rows and pointers allow).  An index outside
// [0, src_rows * div) gives a zero row.  One warp per row.
template <typename V>
__global__ void __launch_bounds__(256) gather_index_kernel(const int* __restrict__ index, int64_t n,
                                                           int div, const V* __restrict__ src,
                                                           int64_t src_rows, int vec_per_row,
                                                           V* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < n;
       r += warps) {
    const int i = __ldg(index + r);
    const int64_t sr = (i >= 0) ? static_cast<int64_t>(i) / div : -1;
    V* d = dst + r * vec_per_row;
    if (sr < 0 || sr >= src_rows) {
      V z;
      memset(&z, 0, sizeof(V));
      for (int c = lane; c < vec_per_row; c += 32) d[c] = z;
    } else {
      const V* sp = src + sr * vec_per_row;
      for (int c = lane; c < vec_per_row; c += 32) d[c] = __ldg(sp + c);
    }
  }
}

// dst[t] = sum_{j < k} (w[t*k+j] or 1) * src[inv[t*k+j]] in fp32, j ascending,
// rows of H elements (H % 8 == 0); a slot whose inv is outside [0, T*k)
// contributes nothing.  One warp per token, 8 elements per lane and step.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) combine_dense_kernel(const Tin* __restrict__ src, int H,
                                                            int k, const int* __restrict__ inv,
                                                            const float* __restrict__ w,
                                                            int64_t T, Tout* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t tk = T * k;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T;
       t += warps) {
    for (int c = lane * 8; c < H; c += 256) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      for (int j = 0; j < k; ++j) {
        const int64_t s = t * k + j;
        const int r = __ldg(inv + s);
        if (r < 0 || r >= tk) continue;
        const float sc = w ? __ldg(w + s) : 1.f;
        float a[8];
        load8(src + static_cast<int64_t>(r) * H + c, a);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(sc, a[i], acc[i]);
      }
      store8(dst + t * H + c, acc);
    }
  }
}

cudaError_t launch_gather_index(const int* index, int64_t n, int div, const void* src,
                                int64_t src_rows, int64_t row_bytes, void* dst, int num_sms,
                                cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t g = std::min<int64_t>((n + 7) / 8, static_cast<int64_t>(num_sms) * 16);
  const bool v16 = (row_bytes % 16 == 0) && (reinterpret_cast<uintptr_t>(src) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(dst) % 16 == 0);
  if (v16)
    gather_index_kernel<<<static_cast<int>(g), 256, 0, st>>>(
        index, n, div, static_cast<const uint4*>(src), src_rows, static_cast<int>(row_bytes / 16),
        static_cast<uint4*>(dst));
  else
    gather_index_kernel<<<static_cast<int>(g), 256, 0, st>>>(
        index, n, div, static_cast<const uint32_t*>(src), src_rows,
        static_cast<int>(row_bytes / 4), static_cast<uint32_t*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_combine_dense(const void* src, int src_bytes, int H, int k, const int* inv,
                                 const float* w, int64_t T, void* dst, int dst_bytes, int num_sms,
                                 cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int g = static_cast<int>(std::min<int64_t>((T + 7) / 8, static_cast<int64_t>(num_sms) * 16));
  using B = __nv_bfloat16;
  if (src_bytes == 2 && dst_bytes == 2)
    combine_dense_kernel<<<g, 256, 0, st>>>(static_cast<const B*>(src), H, k, inv, w, T, static_cast<B*>(dst));
  else if (src_bytes == 2)
    combine_dense_kernel<<<g, 256, 0, st>>>(static_cast<const B*>(src), H, k, inv, w, T, static_cast<float*>(dst));
  else if (dst_bytes == 2)
    combine_dense_kernel<<<g, 256, 0, st>>>(static_cast<const float*>(src), H, k, inv, w, T, static_cast<B*>(dst));
  else
    combine_dense_kernel<<<g, 256, 0, st>>>(static_cast<const float*>(src), H, k, inv, w, T, static_cast<float*>(dst));
  return cudaGetLastError();
}

static int grid_for(int64_t rows, int num_sms) {
  // 8 warps per block; enough blocks to cover every SM several times.
  const int64_t need = (rows + 7) / 8;
  int64_t g = static_cast<int64_t>(num_sms) * 8;
  if (need < g) g = need > 0 ? need : 1;
  return static_cast<int>(g);
}

cudaError_t launch_gather_rows(const void* src, int H, int k, int E, const int* poff,
                               const int* counts, const int* offsets, const int* perm, int tk,
                               int64_t rows_max, void* dst, int elem_bytes, int num_sms,
                               cudaStream_t st) {
  const int vec = H * elem_bytes / 16;
  gather_rows_kernel<<<grid_for(rows_max, num_sms), 256, 0, st>>>(
      static_cast<const uint4*>(src), vec, k, E, poff, counts, offsets, perm, tk, rows_max,
      elem_bytes == 4 ? 1 : 0, static_cast<uint4*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* src, int H, int k, int E, const int* idx, const int* inv,
                           const int* offsets, const int* poff, int64_t T, int64_t rows_max,
                           void* out, int out_bytes, int num_sms, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (k > kMaxK) return cudaErrorInvalidValue;
  if (out_bytes == 2)
    combine_kernel<__nv_bfloat16><<<grid_for(T, num_sms), 256, 0, st>>>(
        src, H, k, E, idx, inv, offsets, poff, T, rows_max, static_cast<__nv_bfloat16*>(out));
  else
    combine_kernel<float><<<grid_for(T, num_sms), 256, 0, st>>>(
        src, H, k, E, idx, inv, offsets, poff, T, rows_max, static_cast<float*>(out));
  return cudaGetLastError();
}

__global__ void __launch_bounds__(256) round_copy_tf32_kernel(const float4* __restrict__ in,
                                                              float4* __restrict__ out, int64_t n4) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = __ldg(in + i);
    out[i] = make_float4(round_tf32(a.x), round_tf32(a.y), round_tf32(a.z), round_tf32(a.w));
  }
}

cudaError_t launch_round_copy_tf32(const float* in, float* out, int64_t n, int num_sms,
                                   cudaStream_t st) {
  const int64_t n4 = n / 4;
  if (n4 == 0) return cudaSuccess;
  int64_t blocks = (n4 + 255) / 256;
  if (blocks > static_cast<int64_t>(num_sms) * 8) blocks = static_cast<int64_t>(num_sms) * 8;
  round_copy_tf32_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(
      reinterpret_cast<const float4*>(in), reinterpret_cast<float4*>(out), n4);
  return cudaGetLastError();
}

cudaError_t launch_transpose_f32(const float* in, float* out, int batch, int rows, int cols,
                                 cudaStream_t st) {
  if (batch == 0 || rows == 0 || cols == 0) return cudaSuccess;
  const int gy = (rows + 31) / 32 < 65535 ? (rows + 31) / 32 : 65535;
  dim3 grid((cols + 31) / 32, gy, batch);
  transpose_f32_kernel<<<grid, dim3(32, 8), 0, st>>>(in, out, rows, cols);
  return cudaGetLastError();
}

cudaError_t launch_dw_reduce(const float* dwpart, int ntiles, int64_t rows_max, int E,
                             const int* idx,
                             const int* inv, const int* offsets, const int* poff, int64_t Tk,
                             float* d_topk_w, cudaStream_t st) {
  if (Tk == 0) return cudaSuccess;
  const int blocks = static_cast<int>((Tk + 255) / 256);
  dw_reduce_kernel<<<blocks, 256, 0, st>>>(dwpart, ntiles, rows_max, E, idx, inv, offsets, poff,
                                           Tk, d_topk_w);
  return cudaGetLastError();
}

cudaError_t launch_bias_slot_dot(const void* dy, const void* b_down, int H, int k, int E,
                                 const int* idx, const int* inv, const int* offsets,
                                 const int* poff, int64_t Tk, int64_t rows_max, float* out,
                                 int elem_bytes, int num_sms, cudaStream_t st) {
  if (Tk == 0) return cudaSuccess;
  const int g = grid_for(Tk, num_sms);
  if (elem_bytes == 2)
    bias_slot_dot_kernel<<<g, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(dy),
                                            static_cast<const __nv_bfloat16*>(b_down), H, k, E,
                                            idx, inv, offsets, poff, Tk, rows_max, out);
  else
    bias_slot_dot_kernel<<<g, 256, 0, st>>>(static_cast<const float*>(dy),
                                            static_cast<const float*>(b_down), H, k, E, idx, inv,
                                            offsets, poff, Tk, rows_max, out);
  return cudaGetLastError();
}

cudaError_t launch_expert_colsum(const void* src, const void* src2, int C, int64_t ld,
                                 int gather_k, int E, const int* poff, const int* counts,
                                 const int* offsets, const int* perm, const float* topk_w, int tk,
                                 bool weighted, const int* src2_flags, float* out, int elem_bytes,
                                 cudaStream_t st) {
  if (C % 8 || E <= 0 || E > 65535) return cudaErrorInvalidValue;
  const dim3 grid((C / 8 + 63) / 64, E), block(64, kRowGroups);
  if (elem_bytes == 2)
    expert_colsum_kernel<<<grid, block, 0, st>>>(
        static_cast<const __nv_bfloat16*>(src), static_cast<const __nv_bfloat16*>(src2), C, ld,
        gather_k, poff, counts, offsets, perm, topk_w, tk, weighted ? 1 : 0, src2_flags, out);
  else
    expert_colsum_kernel<<<grid, block, 0, st>>>(static_cast<const float*>(src),
                                                 static_cast<const float*>(src2), C, ld, gather_k,
                                                 poff, counts, offsets, perm, topk_w, tk,
                                                 weighted ? 1 : 0, src2_flags, out);
  return cudaGetLastError();
}

}  // namespace moe
