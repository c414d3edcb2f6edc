// Internal launchers of the sm_103a kernels (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// ---- dispatch plan (plan.cu)
cudaError_t launch_plan(const int* idx, int64_t Tk, int E, int* counts, int* offsets, int* perm,
                        int* inv, int* poff, int* blkhist, int* err, cudaStream_t st);
cudaError_t launch_padded_offsets(const int* counts, int E, int* poff, cudaStream_t st);
size_t plan_blkhist_ints(int64_t Tk, int E);

// ---- top-k routing (route.cu): topk_idx / topk_w [T,k] from logits [T,E]
// fp32 (finite); ids by descending logit, equal logits by ascending id;
// weights are a softmax over the k chosen logits.  E <= 1024, k <= 32.
cudaError_t launch_route(const float* logits, int64_t T, int E, int k, int* topk_idx,
                         float* topk_w, int num_sms, cudaStream_t st);

// ---- row movement (permute.cu); elem_bytes is 2 (bf16) or 4 (fp32)
// dst[p] = src[perm[offsets[e] + p - poff[e]] / k] for the live rows of the
// tile-padded expert-grouped layout; padding rows (and rows whose slot is
// outside [0, tk)) are zero-filled.  fp32 rows are rounded to TF32 (they are
// TF32 tensor-core operands).
cudaError_t launch_gather_rows(const void* src, int H, int k, int E, const int* poff,
                               const int* counts, const int* offsets, const int* perm, int tk,
                               int64_t rows_max, void* dst, int elem_bytes, int num_sms,
                               cudaStream_t st);
// out[t] = sum_{j<k} src[row(t*k+j)] in fp32, j ascending; k <= 32.  src
// holds fp32 rows [rows_max, H]; out is [T, H] of 2- or 4-byte elements.  A
// slot with an out-of-range expert id contributes nothing.
cudaError_t launch_combine(const float* src, int H, int k, int E, const int* idx, const int* inv,
                           const int* offsets, const int* poff, int64_t T, int64_t rows_max,
                           void* out, int out_bytes, int num_sms, cudaStream_t st);
// out[b][c][r] = round_tf32(in[b][r][c]) for fp32 [batch, rows, cols] arrays.
cudaError_t launch_transpose_f32(const float* in, float* out, int batch, int rows, int cols,
                                 cudaStream_t st);
// out[i] = round_tf32(in[i]), n a multiple of 4.
cudaError_t launch_round_copy_tf32(const float* in, float* out, int64_t n, int num_sms,
                                   cudaStream_t st);
// d_topk_w[s] = sum_{n < ntiles} dwpart[n * rows_max + row(s)], n ascending.
cudaError_t launch_dw_reduce(const float* dwpart, int ntiles, int64_t rows_max, int E,
                             const int* idx,
                             const int* inv, const int* offsets, const int* poff, int64_t Tk,
                             float* d_topk_w, cudaStream_t st);

// ---- per-expert bias terms (permute.cu); elem_bytes 2 (bf16) or 4 (fp32)
// out[row(s)] = <dy[s / k, :H], b_down[idx[s], :H]> for each slot s whose
// padded row row(s) is valid, summed in fp32 in a fixed order.
cudaError_t launch_bias_slot_dot(const void* dy, const void* b_down, int H, int k, int E,
                                 const int* idx, const int* inv, const int* offsets,
                                 const int* poff, int64_t Tk, int64_t rows_max, float* out,
                                 int elem_bytes, int num_sms, cudaStream_t st);
// out[e, c] = sum_{j < counts[e]} s_j * (src[r_j, c] (+ src2[r_j, c])) in fp32,
// in a fixed order; r_j = poff[e] + j, or perm[offsets[e] + j] / gather_k when
// gather_k > 0; s_j = topk_w[perm[offsets[e] + j]] when `weighted`, else 1.
// src / src2 (optional) have row stride ld; C % 8 == 0.  With src2_flags,
// src2 is read only for experts whose flag is non-zero.
cudaError_t launch_expert_colsum(const void* src, const void* src2, int C, int64_t ld,
                                 int gather_k, int E, const int* poff, const int* counts,
                                 const int* offsets, const int* perm, const float* topk_w, int tk,
                                 bool weighted, const int* src2_flags, float* out, int elem_bytes,
                                 cudaStream_t st);
// lo_flags[e] = 0 when expert e's effective row count (sum w^2)^2 / sum w^4
// over its routing weights is at least min_neff (its weight gradients then
// take the computed operand as one bf16 value), else 1 (bf16 hi + lo parts).
cudaError_t launch_split_select(const int* offsets, const int* perm, const float* topk_w, int tk,
                                int E, float min_neff, int* lo_flags, cudaStream_t st);

// ---- dense row movement of the expert-parallel exchange (permute.cu)
// dst[r] = src[index[r] / div] for r < n (rows of row_bytes bytes, a multiple
// of 4); an index outside [0, src_rows * div) gives a zero row.
cudaError_t launch_gather_index(const int* index, int64_t n, int div, const void* src,
                                int64_t src_rows, int64_t row_bytes, void* dst, int num_sms,
                                cudaStream_t st);
// dst[t] = sum_{j<k} (w[t*k+j] or 1) src[inv[t*k+j]] in fp32, j ascending;
// src / dst elements of 2 (bf16) or 4 (fp32) bytes; H % 8 == 0.
cudaError_t launch_combine_dense(const void* src, int src_bytes, int H, int k, const int* inv,
                                 const float* w, int64_t T, void* dst, int dst_bytes, int num_sms,
                                 cudaStream_t st);

// ---- grouped tensor-core GEMMs (gemm_*.cu)
enum GemmMode : int {
  kFwdGateUp = 0,    // A_act = act(Xp Wgu[e]) (+ saved pre-activations)
  kFwdDown = 1,      // Ow = w * (A_act Wd[e])
  kDgradDown = 2,    // dA' = dYp Wd[e]^T -> dH1, Aw, d(topk w) partials
  kDgradGateUp = 3,  // dXp = dH1 Wgu[e]^T
  kWgradDown = 4,    // dWd[e] = Aw^T dYp
  kWgradGateUp = 5   // dWgu[e] = Xp^T dH1
};

// One epilogue output: element (b, r, c) lives at ptr[b*bstride + r*ld + c];
// rows >= rows and columns >= cols are not written.
struct OutDesc {
  void* ptr;
  int64_t ld;
  int64_t bstride;
  int rows;
  int cols;
};

struct GemmArgs {
  const int* poff;      // [E+1] tile-padded row offsets
  const int* counts;    // [E]
  const int* offsets;   // [E+1]
  const int* perm;      // [T*k]
  const float* topk_w;  // [T*k]
  int tk;               // T*k
  int E;
  int n_tiles;          // output-column tiles per expert
  int m_tiles;          // weight-gradient modes: 128-row tiles of the output
  int num_kb;           // row-grouped modes: 128-byte k-blocks of the contraction
  int act;
  int gu_interleaved;   // fused gate_up columns: 0 [gate | up], 1 gate/up interleaved
  float limit;
  float alpha;
  int save_h1;          // kFwdGateUp: also store the gate / up pre-activations
  int h1_half;          // clamped GLU, bf16: the saved pre-activations are fp16 (else fp32)
  const void* bias;     // kFwdGateUp: b_gate_up [E, 2I]; kFwdDown: b_down [E, H]; or null
  const void* h1;       // kDgradDown: saved pre-activations [rows_max, 2I]
  int I;
  float* dwpart;        // kDgradDown: [n_tiles][rows_max]
  const int* lo_flags;  // bf16 backward: per expert, 1 = its weight gradients use the bf16
                        // hi + lo parts of the computed operand, 0 = the hi part alone (the
                        // down dgrad then writes no lo part); null = always both
  int64_t rows_max;
  int* err;
  uint64_t timeout_ns;
  OutDesc out[6];       // mode-specific outputs (see the epilogue)
};

// TMA descriptors of the operands of one GEMM launch (unused ones may repeat
// a valid map):
//   a   A operand (hi part when split)      a2  A lo part (split A); with
//       token-N tiling the token rows' 32-row box (a: 128 rows)
//   b0  B operand (hi part / gate view)     b1  B lo part (split B) / up view
//   out weight gradients: the fp32 dW [E, M, N], box {32, 32}, 128B swizzle
struct GemmMaps {
  CUtensorMap a, a2, b0, b1, out;
};

cudaError_t launch_gemm(int mode, int elem_bytes, const GemmMaps& maps, const GemmArgs& args,
                        int num_sms, cudaStream_t st);
// Column tile width (N) of the output for a mode, as used by launch_gemm.
int gemm_block_n(int mode, int elem_bytes);
int gemm_block_m(int mode, int elem_bytes);

}  // namespace moe
