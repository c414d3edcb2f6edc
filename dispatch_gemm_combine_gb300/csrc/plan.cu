// Dispatch plan: per-expert histogram, prefix scans and the stable
// expert-grouped permutation of the T*k routing slots ("masked indexing" /
// "sparse token extraction" in the pages' descriptions of the layer).
//
// The permutation orders slots by expert id and, within an expert, by slot
// id s = t*k + j, so the plan is unique and the GPU result is bit-exact with
// any correct implementation.
//
// Three launches on the caller's stream:
//   plan_hist     one block per chunk of 1024 slots: chunk-local expert
//                 histogram (shared-memory atomics on integers: exact).
//   plan_scan     one block: per expert, exclusive scan of the chunk
//                 histograms in chunk order (chunk bases), expert counts,
//                 exclusive scan over experts (offsets) and over the
//                 tile-padded counts (padded offsets used by the GEMMs).
//   plan_scatter  one block per chunk: warps of the chunk take turns in
//                 slot order; within a warp, lanes with equal expert id are
//                 ranked by lane (match.any + popc), so every slot gets
//                 base + number of earlier slots of its expert.
#include "kernels.h"

namespace moe {

constexpr int kPlanChunk = 1024;

__global__ void __launch_bounds__(kPlanChunk) plan_hist_kernel(const int* __restrict__ idx,
                                                               int64_t Tk, int E,
                                                               int* __restrict__ blkhist,
                                                               int* __restrict__ err) {
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t s = static_cast<int64_t>(blockIdx.x) * kPlanChunk + threadIdx.x;
  if (s < Tk) {
    const int e = idx[s];
    if (e >= 0 && e < E)
      atomicAdd(&hist[e], 1);
    else
      record_error(err, kErrBadIndex);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    blkhist[static_cast<int64_t>(blockIdx.x) * E + e] = hist[e];
}

// Exclusive scan of one value per thread over a block of 1024 threads.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += y;
    }
    warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  const int excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  if (total) *total = warp_sums[31];
  __syncthreads();
  return excl;
}

// from_counts = 1: counts[] is given (a caller-built plan) and only the
// padded offsets are derived; blkhist is not touched.  poff has 2*(E+1)
// entries: the tile-padded row offsets, then the prefix over experts of
// their number of 128-row tile pairs (the schedule of the 2-SM GEMMs).
__global__ void __launch_bounds__(1024) plan_scan_kernel(int* __restrict__ blkhist, int nchunks,
                                                         int E, int* __restrict__ counts,
                                                         int* __restrict__ offsets,
                                                         int* __restrict__ poff,
                                                         int from_counts) {
  __shared__ int warp_sums[32];
  __shared__ int totals[2];
  const int e = threadIdx.x;
  int c = 0;
  if (e < E) {
    if (from_counts) {
      c = counts[e];
    } else {
      int run = 0;
      for (int b = 0; b < nchunks; ++b) {
        const int64_t i = static_cast<int64_t>(b) * E + e;
        const int h = blkhist[i];
        blkhist[i] = run;
        run += h;
      }
      c = run;
      counts[e] = c;
    }
  }
  int tot = 0;
  const int off = block_exclusive_scan(c, warp_sums, &tot);
  if (threadIdx.x == 0) totals[0] = tot;
  const int padded = (c + kRowTile - 1) / kRowTile * kRowTile;
  int ptot = 0;
  const int pof = block_exclusive_scan(padded, warp_sums, &ptot);
  const int pairs = (padded / kRowTile + 1) / 2;
  int pptot = 0;
  const int ppof = block_exclusive_scan(pairs, warp_sums, &pptot);
  if (e < E) {
    if (!from_counts) offsets[e] = off;
    poff[e] = pof;
    poff[E + 1 + e] = ppof;
  }
  if (threadIdx.x == 0) {
    if (!from_counts) offsets[E] = totals[0];
    poff[E] = ptot;
    poff[E + 1 + E] = pptot;
  }
}

__global__ void __launch_bounds__(kPlanChunk) plan_scatter_kernel(
    const int* __restrict__ idx, int64_t Tk, int E, const int* __restrict__ blkhist,
    const int* __restrict__ offsets, int* __restrict__ perm, int* __restrict__ inv) {
  extern __shared__ int run[];
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    run[e] = offsets[e] + blkhist[static_cast<int64_t>(blockIdx.x) * E + e];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t s = static_cast<int64_t>(blockIdx.x) * kPlanChunk + threadIdx.x;
  int e = -1;
  if (s < Tk) e = idx[s];
  const bool ok = (s < Tk) && e >= 0 && e < E;
  // lanes without a valid slot get a key no other lane has
  const int key = ok ? e : -1 - lane;
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  const int leader = __ffs(peers) - 1;
  const int rank = __popc(peers & ((1u << lane) - 1u));
  for (int w = 0; w < kPlanChunk / 32; ++w) {
    if (warp == w) {
      int base = 0;
      if (ok && lane == leader) {
        base = run[e];
        run[e] = base + __popc(peers);
      }
      base = __shfl_sync(0xffffffffu, base, leader);
      if (ok) {
        const int pos = base + rank;
        perm[pos] = static_cast<int>(s);
        inv[s] = pos;
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_plan(const int* idx, int64_t Tk, int E, int* counts, int* offsets, int* perm,
                        int* inv, int* poff, int* blkhist, int* err, cudaStream_t st) {
  const int nchunks = static_cast<int>((Tk + kPlanChunk - 1) / kPlanChunk);
  const size_t hist_smem = sizeof(int) * static_cast<size_t>(E);
  if (nchunks > 0) {
    plan_hist_kernel<<<nchunks, kPlanChunk, hist_smem, st>>>(idx, Tk, E, blkhist, err);
  }
  plan_scan_kernel<<<1, 1024, 0, st>>>(blkhist, nchunks, E, counts, offsets, poff, 0);
  if (nchunks > 0) {
    plan_scatter_kernel<<<nchunks, kPlanChunk, hist_smem, st>>>(idx, Tk, E, blkhist, offsets,
                                                                perm, inv);
  }
  return cudaGetLastError();
}

cudaError_t launch_padded_offsets(const int* counts, int E, int* poff, cudaStream_t st) {
  plan_scan_kernel<<<1, 1024, 0, st>>>(nullptr, 0, E, const_cast<int*>(counts), nullptr, poff, 1);
  return cudaGetLastError();
}

size_t plan_blkhist_ints(int64_t Tk, int E) {
  const int64_t nchunks = (Tk + kPlanChunk - 1) / kPlanChunk;
  return static_cast<size_t>(nchunks > 0 ? nchunks : 1) * static_cast<size_t>(E);
}

}  // namespace moe
