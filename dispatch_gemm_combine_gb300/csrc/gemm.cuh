// Grouped (per-expert) GEMM on the sm_103a tensor cores: TMA loads into a
// multi-stage shared-memory ring, tcgen05.mma issued by one thread with the
// fp32 accumulator in tensor memory (double-buffered), and a 4-warp epilogue
// that reads the accumulator with tcgen05.ld, applies the mode's fused
// elementwise work and stores through per-warp shared-memory tiles (row
// segments of whole sectors, or TMA tensor stores for the weight gradients).
//
// bf16 kernels use the 2-SM form of the tensor-core MMA (cta_group::2): a
// cluster of two CTAs computes a 256 x N tile.  Each CTA loads its own 128
// rows of A and half (N/2 columns) of B into its shared memory; one thread
// of the even CTA (the leader) issues M=256 MMAs that read both CTAs'
// tiles, and each CTA's tensor memory receives the accumulator rows of its
// own A rows.  A CTA therefore receives 2/3 of the operand bytes per FLOP
// of a single-CTA 128 x N tile (A 16 KB + B 16 KB per k-block for N=256),
// which matters because the operand loads, bounded by the bytes the ring
// keeps in flight, not the MMAs, set the pace of these kernels.  The bf16
// down dgrad, whose epilogue far outweighs its MMAs, and fp32 storage (TF32
// products) use independent CTAs and the 1-SM form.
//
// Warp roles: warp 0 = TMA producer, warp 1 = MMA issuer (in the leader)
// and tensor-memory owner, warps 2..5 = epilogue (warp w reads TMEM lanes
// 32*(w%4) .. 32*(w%4)+31).  Persistent: each CTA pair walks a static
// sequence of work units.
//
// Row-grouped modes (the down dgrad, the interleaved-column gate_up forward
// and the fp32 forward and dgrads) tile the tile-padded expert-grouped row
// space: expert e owns rows [poff[e], poff[e+1]), a multiple of 128, so no
// M tile straddles two experts; a CTA pair takes two consecutive m-tiles of
// one expert, or one m-tile split 64 + 64 (a half unit) for an expert's odd
// last tile.  Token-N modes (the other bf16 forward and dgrad GEMMs) put the
// weights on M and an expert's tokens on N instead, in units of up to 256
// tokens.  Units are ordered (expert, n, m) so the pairs running at the same
// time share one expert's weights in L2.  Weight-gradient modes tile the
// [E, M, N] output (a pair: 256 x N) and contract over the expert's rows,
// stopping at the MMA step that holds its last row (padding rows are
// zero-filled).
//
// Operand layouts (smem, 128-byte swizzle, what TMA writes):
//   K-major   box {128 B of K, rows}: 8-row groups 1024 B apart (SBO); the
//             k-th MMA of a block starts 32*k bytes in.
//   MN-major  boxes {128 B of M or N, BK rows of K}, one per 128 B of M/N,
//             BK*128 B apart (LBO); 8-row K groups 1024 B apart (SBO); the
//             k-th MMA starts k * (MMA K rows) * 128 bytes in.
#pragma once

#include <type_traits>

#include "kernels.h"

namespace moe {

// Limit on the waits that drain copies and MMAs already in flight when a CTA
// unwinds after a timeout; independent of the (adjustable) pipeline limit so
// that a CTA never exits with asynchronous work still writing its memory.
constexpr uint64_t kDrainNs = 1000000000ull;

template <typename T, int MODE, int BN, int STAGES, bool IL_ = false, bool SW_ = false>
struct GemmCfg {
  static constexpr int kES = sizeof(T);
  static constexpr bool kTf32 = (kES == 4);
  static constexpr int BK = 128 / kES;           // elements in one 128-byte row
  static constexpr int CH = 128 / kES;           // MN-major chunk width (elements)
  static constexpr int MMA_K = 32 / kES;         // K of one tcgen05.mma
  static constexpr int KSTEPS = BK / MMA_K;      // MMAs per k-block (4)
  static constexpr bool kWgrad = (MODE == kWgradDown || MODE == kWgradGateUp);
  // interleaved gate_up columns (gate = even, up = odd): a separate
  // instantiation of the two modes that see the layout (the gate_up forward
  // and the down dgrad), so the concatenated kernels are unchanged
  static constexpr bool IL = IL_;
  static_assert(!IL || MODE == kFwdGateUp || MODE == kDgradDown, "layout-specific modes only");
  // Token-N tiling: the weights are the MMA's M operand (128 features per CTA,
  // 256 per pair) and an expert's tokens its N side, in units of up to 256
  // tokens rounded up to 16, so rows that only pad an expert to 128 cost no
  // MMA work.  Used by the bf16 down projection and gate_up dgrad, whose
  // epilogues write fp32 token rows, and by the bf16 gate_up forward with
  // concatenated [gate | up] columns: a CTA's 128 features are the gate and
  // the up columns of the same 64 outputs, so the two warps that hold the
  // gate and the up values of one output pass each other half of a chunk's
  // tokens through shared memory.
  static constexpr bool SW = SW_;
  static_assert(!SW || (sizeof(T) == 2 &&
                        (MODE == kFwdDown || MODE == kDgradGateUp || MODE == kFwdGateUp)),
                "token-N tiling: bf16 down projection, gate_up dgrad and gate_up forward");
  static_assert(!(SW && IL), "token-N tiling of the gate_up forward takes concatenated columns");
  // 2-SM MMA over a CTA pair for every bf16 mode but the down dgrad, whose
  // heavy epilogue would hold up both CTAs (a pair's next MMA waits for both
  // CTAs' epilogues); TF32 keeps independent CTAs
  static constexpr bool CTA2 =
      !kTf32 && (MODE == kFwdGateUp || MODE == kFwdDown || MODE == kDgradGateUp || kWgrad);
  static constexpr int PAIR = CTA2 ? 2 : 1;
  // TF32 operands must be K-major (the fp32 path transposes the others into
  // the workspace first); 16-bit operands may be MN-major.
  static constexpr bool A_MN = (kWgrad || (SW && (MODE == kFwdDown || MODE == kFwdGateUp))) && !kTf32;
  static constexpr bool B_MN = !SW && (MODE == kFwdGateUp || MODE == kFwdDown || kWgrad) && !kTf32;
  // bf16 weight gradients contract a computed operand (w*a, dH1) that the
  // experts with few effectively weighted rows carry as a bf16 hi/lo pair:
  // two MMAs, one per part, into the same accumulator (about 16 bits of
  // mantissa instead of 8).  A k-block of such an expert takes two slots of
  // the shared-memory ring: the operands (hi part) in one, the lo part in
  // the next, each slot with its own barriers; every other k-block takes
  // one, so the ring is as deep as the slots allow.
  static constexpr bool SPLIT_A = (MODE == kWgradDown) && !kTf32;
  static constexpr bool SPLIT_B = (MODE == kWgradGateUp) && !kTf32;
  static constexpr int BN_CTA = BN / PAIR;       // B columns held by one CTA
  static constexpr int A_PART = 128 * 128;       // 128 rows of A, one 128-byte K row each
  static constexpr int B_PART = BN_CTA * 128;
  static constexpr int A_BYTES = A_PART;
  static constexpr int B_BYTES = B_PART;
  static constexpr int LO_BYTES = SPLIT_A ? A_PART : (SPLIT_B ? B_PART : 0);
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // per CTA and ring slot
  static constexpr int CHUNK_BYTES = BK * 128;   // one MN-major box
  // per epilogue warp: one 32x32 transpose tile, rows padded to 36 words;
  // the down dgrad also stages the saved pre-activations of its 32 rows
  // (32 gate + 32 up fp32 per row, rows padded to 68 words)
  // The weight gradients store their fp32 tiles with TMA tensor stores
  // (measured 12% faster than register stores on the down one, 13% on the
  // gate_up one); the fp32 rows of the forward down GEMM and the gate_up
  // dgrad measured within 2% of the shared-memory transposes, so those keep
  // the register paths.
  static constexpr bool TMA_OUT = kWgrad;
  // The producer and the MMA issuer run on one lane (no warp-wide step per
  // k-block), except in the weight gradients, which measured faster with
  // the whole warp stepping through each k-block (their fp32 stores, not
  // the loads, set their pace).
  static constexpr bool kOneLane = !kWgrad;
  static constexpr int H1_WARP_BYTES = (MODE == kDgradDown) ? 32 * 68 * 4 : 0;
  static constexpr int BAR_BYTES = (2 * STAGES + 5) * 8 + 16;
  // TMA_OUT: each epilogue warp stages its stores in STG_BUFS 32 x 32 fp32
  // tiles (128-byte swizzle), as many as the shared memory left beside the
  // ring holds (2 to 6).  A tile may be rewritten only once the store that
  // read it has left shared memory, so the staging bounds the store bytes a
  // warp keeps in flight.
  static constexpr int STG_AVAIL = 232448 - 1024 - STAGES * STAGE_BYTES - BAR_BYTES;
  static constexpr int STG_BUFS =
      STG_AVAIL / (4 * 4096) > 6 ? 6 : (STG_AVAIL / (4 * 4096) < 2 ? 2 : STG_AVAIL / (4 * 4096));
  static constexpr int EPI_WARP_BYTES = TMA_OUT ? STG_BUFS * 4096 : 32 * 36 * 4;
  static constexpr int EPI_BYTES = 4 * (EPI_WARP_BYTES + H1_WARP_BYTES);
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
  static constexpr int ACC_COLS = BN;            // TMEM columns of one tile's accumulator
  static constexpr int TMEM_COLS = (2 * ACC_COLS <= 256) ? 256 : 512;
  // output columns produced per tile (gate_up: BN/2 gate + BN/2 up -> BN/2)
  static constexpr int BN_OUT = (MODE == kFwdGateUp) ? BN / 2 : BN;
  static constexpr uint32_t IDESC = make_idesc(kTf32, A_MN, B_MN, 128 * PAIR, BN);
  // Row-grouped pairs run an expert's odd last m-tile as one M=128 MMA unit
  // instead of an M=256 unit with an idle half.  Each CTA then holds 64 rows;
  // its tensor memory keeps them in lanes 0-63 for columns [0, N/2) and again
  // in lanes 64-127 for columns [N/2, N), in accumulator columns [0, N/2).
  static constexpr uint32_t IDESC_HALF = make_idesc(kTf32, A_MN, B_MN, 128, BN);
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(2 * ACC_COLS <= 512, "two accumulators must fit in tensor memory");
  static_assert(!B_MN || BN_CTA % CH == 0, "MN-major B needs whole chunks");
};

struct TileInfo {
  int e;       // expert
  int row0;    // row-grouped: first padded row of this CTA; wgrad: first padded row of the expert
  int n0;      // first output column
  int m0;      // wgrad: first output row of this CTA
  int nkb;     // k-blocks
  int klast;   // K rows of the last k-block that can be non-zero
  int nt;      // column-tile index
  bool active; // false when this CTA's 128 rows lie past the expert (or the output)
  bool half;   // row-grouped pair unit of one 128-row tile (64 rows per CTA, M = 128)
  int nn;      // token-N tiling: tokens (N) of this unit, a multiple of 16
  bool lo;     // bf16 backward: this expert's computed operand carries its bf16 remainder
};

// Work unit t of the schedule.  A unit is PAIR consecutive m-tiles with one
// column tile; CTA `rank` of the pair takes m-tile unit_m*PAIR+rank (of
// 128 output rows for the weight gradients).  In row-grouped pairs, the
// last unit of an expert with an odd number of m-tiles is a half unit: its
// one m-tile is split into 64 rows per CTA.
template <int BN_OUT, bool kWgrad, int PAIR, bool SW = false>
__device__ __forceinline__ TileInfo decode_tile(const GemmArgs& a, int t, int bk, int rank) {
  TileInfo ti;
  ti.half = false;
  ti.nn = 0;
  ti.lo = true;
  const int NT = a.n_tiles;
  if constexpr (kWgrad) {
    const int MP = (a.m_tiles + PAIR - 1) / PAIR;
    const int per_e = MP * NT;
    ti.e = t / per_e;
    if (a.lo_flags) ti.lo = __ldg(a.lo_flags + ti.e) != 0;
    const int r = t - ti.e * per_e;
    const int mp = r / NT;
    ti.nt = r - mp * NT;
    const int m = mp * PAIR + rank;
    ti.m0 = m * 128;
    ti.active = m < a.m_tiles;
    ti.row0 = __ldg(a.poff + ti.e);
    // contract over the expert's rows only, not over its zero padding: the
    // k-blocks that hold rows, and in the last of them the MMAs that do
    const int cnt = min(__ldg(a.counts + ti.e), __ldg(a.poff + ti.e + 1) - ti.row0);
    ti.nkb = (cnt + bk - 1) / bk;
    ti.klast = cnt - (ti.nkb - 1) * bk;
  } else {
    // unit prefix of expert e: its tile pairs (PAIR = 2) or tiles (PAIR = 1)
    const int* up = (PAIR == 2) ? a.poff + a.E + 1 : a.poff;
    const int sh = (PAIR == 2) ? 0 : 7;
    int lo = 0, hi = a.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((__ldg(up + mid) >> sh) * NT <= t)
        lo = mid;
      else
        hi = mid - 1;
    }
    ti.e = lo;
    if (a.lo_flags) ti.lo = __ldg(a.lo_flags + lo) != 0;
    const int p0 = __ldg(a.poff + lo);
    const int mt = (__ldg(a.poff + lo + 1) - p0) >> 7;
    const int mu = ((__ldg(up + lo + 1) - __ldg(up + lo)) >> sh);   // units of m
    const int local = t - (__ldg(up + lo) >> sh) * NT;
    ti.nt = local / mu;
    const int mp = local - ti.nt * mu;
    if constexpr (SW) {
      // token unit mp of the expert (mu = ceil(count / 256) of them): tokens
      // [256 mp, min(count, 256 mp + 256)), N rounded up to 16; the pair's
      // two CTAs hold its first and second N/2 token rows
      const int left = __ldg(a.counts + lo) - mp * 256;
      ti.nn = ((min(left, 256) + 15) >> 4) << 4;
      ti.row0 = p0 + mp * 256;
      ti.active = left > 0;
      ti.m0 = 0;
      ti.nkb = a.num_kb;
      ti.klast = bk;
      ti.n0 = ti.nt * BN_OUT;
      return ti;
    }
    const int m = mp * PAIR + rank;
    ti.active = m < mt;
    ti.row0 = p0 + m * 128;
    if (PAIR == 2 && (mt & 1) && mp == mu - 1) {
      ti.half = true;
      ti.active = true;
      ti.row0 = p0 + (mt - 1) * 128 + rank * 64;
    }
    ti.m0 = 0;
    ti.nkb = a.num_kb;
    ti.klast = bk;
  }
  ti.n0 = ti.nt * BN_OUT;
  return ti;
}

// The activation is a template parameter so that the unrolled per-element
// loops of the epilogues carry no branch: ACT 0 = SwiGLU, 1 = clamped GLU.
template <int ACT>
__device__ __forceinline__ float act_fwd(float g, float u, float L, float alpha) {
  if constexpr (ACT == 0) return g * sigmoidf_(g) * u;
  const float gc = fminf(g, L);
  const float uc = fminf(fmaxf(u, -L), L);
  return (uc + 1.f) * gc * sigmoidf_(alpha * gc);
}

// a, da/dg, da/du (inclusive clamp masks)
template <int ACT>
__device__ __forceinline__ void act_bwd(float g, float u, float L, float alpha, float& a,
                                        float& dg, float& du) {
  if constexpr (ACT == 0) {
    const float s = sigmoidf_(g);
    const float sg = g * s;
    a = sg * u;
    dg = u * s * (1.f + g * (1.f - s));
    du = sg;
  } else {
    const float gc = fminf(g, L);
    const float uc = fminf(fmaxf(u, -L), L);
    const float s = sigmoidf_(alpha * gc);
    const float glu = gc * s;
    a = (uc + 1.f) * glu;
    dg = (g <= L) ? (uc + 1.f) * (s + alpha * gc * s * (1.f - s)) : 0.f;
    du = (u >= -L && u <= L) ? glu : 0.f;
  }
}

// act_bwd for two elements at once on the packed fp32 pipe (two-wide fma,
// add and mul; the comparisons, clamps and the exponential stay scalar).
// The clamped GLU's ds/dg is written s (1 + alpha gc (1 - s)), the same
// quantity as s + alpha gc s (1 - s).
template <int ACT>
__device__ __forceinline__ void act_bwd2(float2 g, float2 u, float L, float alpha, float2& a,
                                         float2& dg, float2& du) {
  const float2 one = make_float2(1.f, 1.f), mone = make_float2(-1.f, -1.f);
  if constexpr (ACT == 0) {
    const float2 s = make_float2(sigmoidf_(g.x), sigmoidf_(g.y));
    const float2 sg = __fmul2_rn(g, s);
    a = __fmul2_rn(sg, u);
    const float2 oms = __ffma2_rn(s, mone, one);                    // 1 - s
    dg = __fmul2_rn(__fmul2_rn(u, s), __ffma2_rn(g, oms, one));     // u s (1 + g (1 - s))
    du = sg;
  } else {
    const float2 gc = make_float2(fminf(g.x, L), fminf(g.y, L));
    const float2 uc = make_float2(fminf(fmaxf(u.x, -L), L), fminf(fmaxf(u.y, -L), L));
    const float2 ag = __fmul2_rn(gc, make_float2(alpha, alpha));
    const float2 s = make_float2(sigmoidf_(ag.x), sigmoidf_(ag.y));
    const float2 glu = __fmul2_rn(gc, s);
    const float2 up1 = __fadd2_rn(uc, one);
    a = __fmul2_rn(up1, glu);
    const float2 oms = __ffma2_rn(s, mone, one);
    const float2 d = __fmul2_rn(up1, __fmul2_rn(s, __ffma2_rn(ag, oms, one)));
    dg = make_float2(g.x <= L ? d.x : 0.f, g.y <= L ? d.y : 0.f);
    du = make_float2((u.x >= -L && u.x <= L) ? glu.x : 0.f, (u.y >= -L && u.y <= L) ? glu.y : 0.f);
  }
}

// Two fp32 values as one 32-bit pair of the 16-bit output type (round to
// nearest).
template <typename O>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Store this warp's 32x32 output tile: lane i holds row r0+i, columns
// [c0, c0+32).  The tile goes through a per-warp shared-memory transpose,
// then every store instruction writes whole rows: 8 lanes x 16 B = one
// 128-byte fp32 row segment, or 4 lanes x 16 B = one 64-byte 16-bit row
// segment.  Both the row-wise writes and the segment-wise reads are free of
// bank conflicts: fp32 rows are padded to 36 words; 16-bit rows are 64 bytes
// (four 16-byte chunks) with chunk j of row i at position j ^ ((i >> 1) & 3),
// so any 8 rows' chunk j (a write wavefront) and any 2 rows' 4 chunks (a read
// wavefront) fall in 8 different 16-byte bank groups.  Rows >= o.rows and
// columns >= o.cols are not written.
template <typename O>
__device__ __forceinline__ void store_tile(const OutDesc& o, int b, int r0, int c0,
                                           const float (&v)[32], uint8_t* stage, int lane) {
  O* base = static_cast<O*>(o.ptr) + static_cast<int64_t>(b) * o.bstride;
  if constexpr (sizeof(O) == 4) {
    float* st = reinterpret_cast<float*>(stage);
    float* row = st + lane * 36;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<float4*>(row + 4 * j) =
          make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    __syncwarp();
    const int c = (lane & 7) * 4;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int r = it * 4 + (lane >> 3);
      const float4 val = *reinterpret_cast<const float4*>(st + r * 36 + c);
      const int gr = r0 + r, gc = c0 + c;
      if (gr < o.rows && gc < o.cols)
        *reinterpret_cast<float4*>(base + static_cast<int64_t>(gr) * o.ld + gc) = val;
    }
    __syncwarp();
  } else {
    uint4* st = reinterpret_cast<uint4*>(stage);   // [32 rows][4 chunks of 16 B]
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 pk = make_uint4(pack2<O>(v[8 * j], v[8 * j + 1]), pack2<O>(v[8 * j + 2], v[8 * j + 3]),
                                  pack2<O>(v[8 * j + 4], v[8 * j + 5]),
                                  pack2<O>(v[8 * j + 6], v[8 * j + 7]));
      st[lane * 4 + (j ^ sw)] = pk;
    }
    __syncwarp();
    const int c = (lane & 3) * 8;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int r = it * 8 + (lane >> 2);
      const uint4 val = st[r * 4 + ((lane & 3) ^ ((r >> 1) & 3))];
      const int gr = r0 + r, gc = c0 + c;
      if (gr < o.rows && gc < o.cols)
        *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(base) +
                                  static_cast<int64_t>(gr) * o.ld + gc) = val;
    }
    __syncwarp();
  }
}

// Store a 32 x 32 fp32 tile held by columns (lane i holds column c0 + i of
// rows r0 .. r0+31 in v[0..31]): the per-warp stage transposes it, then each
// store writes whole 128-byte row segments, row r scaled by rs(r).  Rows >=
// nrows and columns >= o.cols are not written.
template <typename F>
__device__ __forceinline__ void store_tile_t(const OutDesc& o, int r0, int c0,
                                             const float (&v)[32], uint8_t* stage, int lane,
                                             int nrows, F&& rs) {
  float* base = static_cast<float*>(o.ptr);
  float* st = reinterpret_cast<float*>(stage);
#pragma unroll
  for (int j = 0; j < 32; ++j) st[j * 36 + lane] = v[j];
  __syncwarp();
  const int c = (lane & 7) * 4;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int r = it * 4 + (lane >> 3);
    float4 val = *reinterpret_cast<const float4*>(st + r * 36 + c);
    const float sc = rs(r);
    val.x *= sc;
    val.y *= sc;
    val.z *= sc;
    val.w *= sc;
    const int gc = c0 + c;
    if (r < nrows && gc < o.cols)
      *reinterpret_cast<float4*>(base + static_cast<int64_t>(r0 + r) * o.ld + gc) = val;
  }
  __syncwarp();
}

// Stage lane r's 32 fp32 values as row r of a 32 x 32 tile in the 128-byte
// swizzle at `buf` (1024-byte aligned; conflict-free 16-byte stores) and
// store the tile at (x, y, z) of `map` with one TMA tensor store issued by
// lane 0.  Callers cycle through NBUF buffers, one bulk group per use: the
// wait leaves at most NBUF - 1 later groups reading shared memory, so the
// last store from `buf` has read it.
template <int NBUF>
__device__ __forceinline__ void tma_store_tile32(const CUtensorMap* map, uint32_t buf,
                                                 const float* v, int x, int y, int z, int lane) {
  if (lane == 0) bulk_wait_read<NBUF - 1>();
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 8; ++j)
    st_shared_v4(buf + lane * 128 + ((j ^ (lane & 7)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                 v[4 * j + 3]);
  fence_async_shared();
  __syncwarp();
  if (lane == 0) {
    tma_store_3d(map, buf, x, y, z);
    bulk_commit();
  }
}

// Store n (16 or 32) rows of a tile held by columns as 16-bit values: lane
// i holds column c0 + i of rows r0 .. r0+n-1 in v[0..n-1].  The per-warp
// stage holds n rows of 64 bytes (each lane writes its 2-byte value of every
// row: 64 contiguous bytes per instruction), then every store writes a
// whole 64-byte row segment (4 lanes x 16 B; a read wavefront of 8 lanes
// covers two consecutive rows, 128 contiguous bytes).  Rows >= nrows and
// columns >= o.cols (a multiple of 8) are not written.
template <typename O, int N>
__device__ __forceinline__ void store_tile_t16(const OutDesc& o, int r0, int c0, const float* v,
                                               uint8_t* stage, int lane, int nrows) {
  O* st = reinterpret_cast<O*>(stage);
#pragma unroll
  for (int j = 0; j < N; ++j) {
    if constexpr (std::is_same<O, __half>::value)
      st[j * 32 + lane] = __float2half_rn(v[j]);
    else
      st[j * 32 + lane] = __float2bfloat16_rn(v[j]);
  }
  __syncwarp();
  O* base = static_cast<O*>(o.ptr);
  const int c = (lane & 3) * 8;
  const uint4* s4 = reinterpret_cast<const uint4*>(stage);
#pragma unroll
  for (int it = 0; it < N / 8; ++it) {
    const int r = it * 8 + (lane >> 2);
    const uint4 val = s4[r * 4 + (lane & 3)];
    if (r < nrows && c0 + c < o.cols)
      *reinterpret_cast<uint4*>(base + static_cast<int64_t>(r0 + r) * o.ld + c0 + c) = val;
  }
  __syncwarp();
}

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

__device__ __forceinline__ void split_bf16(float x, float& hi, float& lo) {
  hi = bf16_round(x);
  lo = x - hi;
}

// The clamped GLU's saved pre-activations may be fp16 (bf16 storage, a clamp
// limit L that fp16 represents exactly, |L| <= 32768; the host decides):
// the backward needs gc = min(g, L), uc = clamp(u, -L, L) and the masks
// [g <= L], [-L <= u <= L].  A value past its clamp is kept as an infinite
// marker (it decodes to the clamp with mask 0); a value inside rounds to the
// nearest fp16 value, which stays inside because L is an fp16 value, so
// every mask is exact.  g below -65504 is kept as -65504: the activation and
// its derivatives there are the fp32 results at any such g (sigmoid(alpha g)
// underflows to 0 for alpha >= 0.002).  NaN stays NaN.  The fp16 store does
// the rounding.
__device__ __forceinline__ float h1_code_gate(float g, float L) {
  return g > L ? __int_as_float(0x7f800000) : (g < -65504.f ? -65504.f : g);
}
__device__ __forceinline__ float h1_code_up(float u, float L) {
  return u > L ? __int_as_float(0x7f800000) : (u < -L ? __int_as_float(0xff800000) : u);
}

// Add the bias values p[0, N) of a column chunk to v: every lane of the warp
// reads the same addresses (the chunk's columns are shared by the warp's
// rows), so each 16-byte load is one broadcast.  Only p[0, n) exists (n a
// multiple of 16 bytes' worth of elements); the rest belong to columns past
// the output, which are not stored, and are left out.  p is 16-byte aligned.
template <typename T, int N>
__device__ __forceinline__ void add_bias(const T* p, int n, float (&v)[N]) {
  constexpr int PER = 16 / static_cast<int>(sizeof(T));
#pragma unroll
  for (int j = 0; j < N / PER; ++j) {
    if (j * PER < n) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(p) + j);
      if constexpr (sizeof(T) == 2) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(h[i]);
          v[8 * j + 2 * i] += f.x;
          v[8 * j + 2 * i + 1] += f.y;
        }
      } else {
        v[4 * j] += __uint_as_float(q.x);
        v[4 * j + 1] += __uint_as_float(q.y);
        v[4 * j + 2] += __uint_as_float(q.z);
        v[4 * j + 3] += __uint_as_float(q.w);
      }
    }
  }
}

template <typename T, int MODE, int BN, int STAGES, bool IL, bool SW>
__global__ void __launch_bounds__(192, 1)
    moe_gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmArgs args) {
  using C = GemmCfg<T, MODE, BN, STAGES, IL, SW>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  const uint32_t s_stages = sbase;
  uint8_t* epi_g = gbase + STAGES * C::STAGE_BYTES;
  const uint32_t bars = sbase + STAGES * C::STAGE_BYTES + C::EPI_BYTES;
  const uint32_t full_bar = bars;                    // [STAGES]
  const uint32_t empty_bar = bars + 8 * STAGES;      // [STAGES]
  const uint32_t tfull_bar = bars + 16 * STAGES;     // [2]
  const uint32_t tempty_bar = tfull_bar + 16;        // [2]
  const uint32_t drain_bar = tempty_bar + 16;        // [1] end of the MMA stream
  const uint32_t tmem_slot = drain_bar + 8;
  volatile uint32_t* tmem_slot_g =
      reinterpret_cast<volatile uint32_t*>(gbase + (tmem_slot - sbase));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // rank in the CTA pair; the even CTA issues the MMAs of both
  const int crank = C::CTA2 ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = (crank == 0);
  constexpr uint16_t kPairMask = 0x3;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar + 8 * s, 1);
      mbar_init(empty_bar + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(tfull_bar + 8 * s, 1);
      mbar_init(tempty_bar + 8 * s, 4 * C::PAIR);   // one lane of every epilogue warp of the pair
    }
    mbar_init(drain_bar, 1);
    fence_barrier_init();
    prefetch_tmap(&maps.a);
    prefetch_tmap(&maps.b0);
  }
  if (warp == 1) {
    if constexpr (C::CTA2) {
      tmem_alloc2(tmem_slot, C::TMEM_COLS);
      tmem_relinquish2();
    } else {
      tmem_alloc(tmem_slot, C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (C::CTA2) cluster_sync();   // both CTAs' barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot_g;

  // The leader's barriers receive the TMA completions of both CTAs and the
  // accumulator releases of both epilogues.
  auto leader_addr = [&](uint32_t a) -> uint32_t { return C::CTA2 ? mapa_shared(a, 0) : a; };

  int total;
  if constexpr (C::kWgrad) {
    total = args.E * ((args.m_tiles + C::PAIR - 1) / C::PAIR) * args.n_tiles;
  } else {
    // never past the workspace bound, even for an inconsistent caller plan
    const int rows = static_cast<int>(
        min(static_cast<int64_t>(__ldg(args.poff + args.E)), args.rows_max));
    const int units = (C::PAIR == 2) ? (rows == __ldg(args.poff + args.E)
                                            ? __ldg(args.poff + 2 * args.E + 1)
                                            : 0)
                                     : (rows >> 7);
    total = units * args.n_tiles;
  }
  const int unit0 = blockIdx.x / C::PAIR;
  const int ustride = gridDim.x / C::PAIR;
  const uint64_t tmo = args.timeout_ns;
  // next slot of the shared-memory ring; the barrier parity flips per lap
  auto ring_next = [](int& s, uint32_t& p) {
    if (++s == STAGES) {
      s = 0;
      p ^= 1u;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // (one lane issues everything unless the mode keeps the whole warp in
    // step, see GemmCfg::kOneLane)
    if (!C::kOneLane || lane == 0) {
    // the leader's full barriers, which count the bytes of both CTAs
    const uint32_t full_bar_l = leader_addr(full_bar);
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int t = unit0; t < total && ok; t += ustride) {
      const TileInfo ti = decode_tile<C::BN_OUT, C::kWgrad, C::PAIR, C::SW>(args, t, C::BK, crank);
      // a split operand's expert: the lo part of each k-block in the next slot
      const bool two = C::LO_BYTES > 0 && ti.lo;
      for (int kb = 0; kb < ti.nkb; ++kb) {
        int stage2 = stage;
        uint32_t phase2 = phase;
        if (two) ring_next(stage2, phase2);
        int good = 1;
        if (lane == 0) {
          good = mbar_wait(empty_bar + 8 * stage, phase ^ 1u, tmo);
          if (good && two) good = mbar_wait(empty_bar + 8 * stage2, phase2 ^ 1u, tmo);
        }
        if constexpr (!C::kOneLane) good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          if (lane == 0) record_error(args.err, kErrTimeout);
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t fb = full_bar + 8 * stage;
          const uint32_t fbt = full_bar_l + 8 * stage;
          const uint32_t sA = s_stages + stage * C::STAGE_BYTES;
          const uint32_t sB = sA + C::A_BYTES;
          // the lo part's slot (two-slot k-blocks)
          const uint32_t fb2 = full_bar + 8 * stage2;
          const uint32_t fbt2 = full_bar_l + 8 * stage2;
          const uint32_t sA2 = s_stages + stage2 * C::STAGE_BYTES;
          const uint32_t sB2 = sA2 + C::A_BYTES;
          // token-N tiling: a unit of at most 64 tokens (32 rows per CTA)
          // loads its token rows with the 32-row box of maps.a2
          const bool small_b = C::SW && ti.nn <= 64;
          const uint32_t stage_tx = small_b ? C::A_BYTES + 32 * 128 : C::STAGE_BYTES;
          // the leader expects the bytes of both CTAs of the pair
          if (leader) {
            mbar_arrive_expect_tx(fb, C::PAIR * stage_tx);
            if (two) mbar_arrive_expect_tx(fb2, C::PAIR * C::LO_BYTES);
          }
          auto load2 = [&](uint32_t dst, const CUtensorMap* m, int c0, int c1, uint32_t bar = 0) {
            if (bar == 0) bar = fbt;
            if constexpr (C::CTA2)
              tma_load_2d_g2(dst, m, bar, c0, c1);
            else
              tma_load_2d(dst, m, bar, c0, c1);
          };
          auto load3 = [&](uint32_t dst, const CUtensorMap* m, int c0, int c1, int c2) {
            if constexpr (C::CTA2)
              tma_load_3d_g2(dst, m, fbt, c0, c1, c2);
            else
              tma_load_3d(dst, m, fbt, c0, c1, c2);
          };
          const int kc = kb * C::BK;
          if constexpr (C::SW) {
            // A: this CTA's 128 features of the expert's weights (maps.b0);
            // B: this CTA's half of the unit's token rows (maps.a)
            const int f0 = ti.n0 + crank * 128;
            if constexpr (MODE == kFwdGateUp) {
              // the gate and the up columns of this CTA's 64 outputs
              const int g0 = ti.n0 + crank * C::CH;
              load3(sA, &maps.b0, g0, kc, ti.e);
              load3(sA + C::CHUNK_BYTES, &maps.b1, g0, kc, ti.e);
            } else if constexpr (C::A_MN) {
#pragma unroll
              for (int c = 0; c < 128 / C::CH; ++c)
                load3(sA + c * C::CHUNK_BYTES, &maps.b0, f0 + c * C::CH, kc, ti.e);
            } else {
              load3(sA, &maps.b0, kc, f0, ti.e);
            }
            load2(sB, small_b ? &maps.a2 : &maps.a, kc, ti.row0 + crank * (ti.nn >> 1));
          } else {
          // ---- A: this CTA's 128 rows
          if constexpr (C::kWgrad && !C::A_MN) {
            load2(sA, &maps.a, ti.row0 + kc, ti.m0);   // K-major (transposed) activations
          } else if constexpr (!C::A_MN) {
            load2(sA, &maps.a, kc, ti.row0);
          } else {
            // MN-major chunks (128 B of M x BK rows); a split A's lo part in
            // the next slot
#pragma unroll
            for (int c = 0; c < 128 / C::CH; ++c)
              load2(sA + c * C::CHUNK_BYTES, &maps.a, ti.m0 + c * C::CH, ti.row0 + kc);
            if (C::SPLIT_A && two) {
#pragma unroll
              for (int c = 0; c < 128 / C::CH; ++c)
                load2(sA2 + c * C::CHUNK_BYTES, &maps.a2, ti.m0 + c * C::CH, ti.row0 + kc, fbt2);
            }
          }
          // ---- B: this CTA's BN_CTA columns
          const int nb = ti.n0 + crank * C::BN_CTA;
          if constexpr (MODE == kFwdGateUp && C::B_MN) {
            // bf16 row-grouped gate_up (interleaved columns; concatenated
            // ones tile tokens on N): each CTA of the pair holds the gate and
            // the up columns of the same 64 outputs, the 128 consecutive
            // columns 2*(n0 + 64*rank) ... of the view of all 2I columns, so
            // that a half unit's lanes still see gate and up of one output
            // side by side
            static_assert(C::IL, "bf16 concatenated gate_up columns tile tokens on N");
            static_assert(C::BN_CTA == 2 * C::CH, "gate_up pair tile: one gate and one up chunk per CTA");
            const int col = 2 * (ti.n0 + crank * C::CH);
            load3(sB, &maps.b0, col, kc, ti.e);
            load3(sB + C::CHUNK_BYTES, &maps.b0, col + C::CH, kc, ti.e);
          } else if constexpr (MODE == kFwdGateUp) {
            // K-major (transposed) weights: gate rows then up rows of the tile
            load3(sB, &maps.b0, kc, ti.n0, ti.e);
            load3(sB + (BN / 2) * 128, &maps.b1, kc, ti.n0, ti.e);
          } else if constexpr (MODE == kFwdDown && C::B_MN) {
#pragma unroll
            for (int c = 0; c < C::BN_CTA / C::CH; ++c)
              load3(sB + c * C::CHUNK_BYTES, &maps.b0, nb + c * C::CH, kc, ti.e);
          } else if constexpr (!C::kWgrad) {
            load3(sB, &maps.b0, kc, nb, ti.e);   // K-major weights, box {BK, BN_CTA}
          } else if constexpr (!C::B_MN) {
            load2(sB, &maps.b0, ti.row0 + kc, nb);
          } else {
#pragma unroll
            for (int c = 0; c < C::BN_CTA / C::CH; ++c)
              load2(sB + c * C::CHUNK_BYTES, &maps.b0, nb + c * C::CH, ti.row0 + kc);
            if (C::SPLIT_B && two) {   // a split B's lo part in the next slot
#pragma unroll
              for (int c = 0; c < C::BN_CTA / C::CH; ++c)
                load2(sB2 + c * C::CHUNK_BYTES, &maps.b1, nb + c * C::CH, ti.row0 + kc, fbt2);
            }
          }
          }
        }
        if constexpr (!C::kOneLane) __syncwarp();
        // (each slot used counts once: the drain below waits for every use)
        issued += two ? 2 : 1;
        ring_next(stage, phase);
        if (two) ring_next(stage, phase);
      }
    }
    // Before the CTAs may exit, every load issued must have landed: the
    // leader's full barriers count the bytes of both CTAs.
    if (lane == 0 && leader) {
      for (int s = 0; s < STAGES; ++s) {
        const int64_t n_s = (issued > s) ? (issued - 1 - s) / STAGES + 1 : 0;
        if (n_s > 0 &&
            !mbar_wait(full_bar + 8 * s, static_cast<uint32_t>((n_s - 1) & 1), kDrainNs))
          record_error(args.err, kErrTimeout);
      }
    }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && (!C::kOneLane || lane == 0)) {   // (one lane, see GemmCfg::kOneLane)
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = unit0; t < total && ok; t += ustride) {
        const TileInfo ti = decode_tile<C::BN_OUT, C::kWgrad, C::PAIR, C::SW>(args, t, C::BK, crank);
        int good = 1;
        if (lane == 0) good = mbar_wait(tempty_bar + 8 * acc, acc_phase ^ 1u, tmo);
        if constexpr (!C::kOneLane) good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          if (lane == 0) record_error(args.err, kErrTimeout);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * C::ACC_COLS;
        const bool two = C::LO_BYTES > 0 && ti.lo;   // (as in the producer)
        const uint32_t unit_idesc = C::SW ? make_idesc(C::kTf32, C::A_MN, C::B_MN, 256, ti.nn)
                                          : (ti.half ? C::IDESC_HALF : C::IDESC);
        for (int kb = 0; kb < ti.nkb; ++kb) {
          int stage2 = stage;
          uint32_t phase2 = phase;
          if (two) ring_next(stage2, phase2);
          if (lane == 0) {
            good = mbar_wait(full_bar + 8 * stage, phase, tmo);
            if (good && two) good = mbar_wait(full_bar + 8 * stage2, phase2, tmo);
          }
          if constexpr (!C::kOneLane) good = __shfl_sync(0xffffffffu, good, 0);
          if (!good) {
            if (lane == 0) record_error(args.err, kErrTimeout);
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t sA = s_stages + stage * C::STAGE_BYTES;
            const uint32_t sB = sA + C::A_BYTES;
            const uint32_t sA2 = s_stages + stage2 * C::STAGE_BYTES;   // lo part (two slots)
            const uint32_t sB2 = sA2 + C::A_BYTES;
            const uint32_t idesc = unit_idesc;
            auto mma = [&](uint64_t ad, uint64_t bd, uint32_t accum) {
              if constexpr (C::CTA2)
                tc_mma2(d_tmem, ad, bd, idesc, accum);
              else
                tc_mma<C::kTf32>(d_tmem, ad, bd, C::IDESC, accum);
            };
            // MMAs of this k-block (the last one of a weight gradient may
            // end early)
            const int ksteps = (kb + 1 == ti.nkb) ? (ti.klast + C::MMA_K - 1) / C::MMA_K : C::KSTEPS;
#pragma unroll
            for (int kk = 0; kk < C::KSTEPS; ++kk) {
              if (kk >= ksteps) break;
              const uint32_t aoff = C::A_MN ? kk * C::MMA_K * 128 : kk * 32;
              const uint32_t boff = C::B_MN ? kk * C::MMA_K * 128 : kk * 32;
              const uint32_t albo = C::A_MN ? C::CHUNK_BYTES : 16;
              const uint32_t blbo = C::B_MN ? C::CHUNK_BYTES : 16;
              const uint64_t adesc = smem_desc_sw128(sA + aoff, albo, 1024);
              const uint64_t bdesc = smem_desc_sw128(sB + boff, blbo, 1024);
              mma(adesc, bdesc, (kb | kk) != 0 ? 1u : 0u);
              if constexpr (C::SPLIT_A)
                if (two) mma(smem_desc_sw128(sA2 + aoff, albo, 1024), bdesc, 1u);
              if constexpr (C::SPLIT_B)
                if (two) mma(adesc, smem_desc_sw128(sB2 + boff, blbo, 1024), 1u);
            }
            // the slots are free in both CTAs once these MMAs have read them
            if constexpr (C::CTA2) {
              tc_commit2_mc(empty_bar + 8 * stage, kPairMask);
              if (two) tc_commit2_mc(empty_bar + 8 * stage2, kPairMask);
            } else {
              tc_commit(empty_bar + 8 * stage);
              if (two) tc_commit(empty_bar + 8 * stage2);
            }
          }
          if constexpr (!C::kOneLane) __syncwarp();
          ring_next(stage, phase);
          if (two) ring_next(stage, phase);
        }
        if (!ok) break;
        if (lane == 0) {
          if (ti.nkb > 0) {
            if constexpr (C::CTA2)
              tc_commit2_mc(tfull_bar + 8 * acc, kPairMask);
            else
              tc_commit(tfull_bar + 8 * acc);
          } else {
            // nothing to accumulate (an expert without rows): zeros are stored
            mbar_arrive(tfull_bar + 8 * acc);
            if constexpr (C::CTA2) mbar_arrive_cluster(mapa_shared(tfull_bar + 8 * acc, 1));
          }
        }
        if constexpr (!C::kOneLane) __syncwarp();
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // End of the MMA stream (also after a timeout): one more commit
      // arrives on the drain barrier of both CTAs once every MMA and every
      // stage release issued before it has completed.
      if (lane == 0) {
        if constexpr (C::CTA2)
          tc_commit2_mc(drain_bar, kPairMask);
        else
          tc_commit(drain_bar);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                 // TMEM lane quarter = tile rows q*32..q*32+31
    uint8_t* my_epi = epi_g + (warp - 2) * (C::EPI_WARP_BYTES + C::H1_WARP_BYTES);
    uint8_t* my_h1 = my_epi + C::EPI_WARP_BYTES;
    int acc = 0;
    uint32_t acc_phase = 0;
    // TMA_OUT staging: the next of this warp's STG_BUFS 32 x 32 fp32 tiles
    uint32_t stg_next = 0;
    auto stg_buf = [&]() -> uint32_t {
      const uint32_t b = smem_u32(my_epi) + stg_next * 4096;
      stg_next = (stg_next + 1 == C::STG_BUFS) ? 0u : stg_next + 1;
      return b;
    };

    for (int t = unit0; t < total; t += ustride) {
      const TileInfo ti = decode_tile<C::BN_OUT, C::kWgrad, C::PAIR, C::SW>(args, t, C::BK, crank);
      int good = 1;
      if (lane == 0) good = mbar_wait(tfull_bar + 8 * acc, acc_phase, tmo);
      good = __shfl_sync(0xffffffffu, good, 0);
      // the token-N gate_up forward's warp pairs meet at named barriers:
      // both warps of a pair go on only if both saw the accumulator
      if constexpr (C::SW && MODE == kFwdGateUp) good = pair_and(1 + (q & 1), good != 0) ? 1 : 0;
      if (!good) {
        if (lane == 0) record_error(args.err, kErrTimeout);
        break;
      }
      tc_fence_after();
      // Row-grouped modes: a warp whose 32 rows all lie in the expert's
      // padding has nothing to produce.  Those rows are read later only as
      // rows of other row-grouped GEMMs (whose results for them are ignored),
      // never by the combine, the routing-weight reduction or the weight
      // gradients (whose last MMA step ends inside the warp holding the
      // expert's last row).
      // first tile row of this warp: a half unit's 64 rows per CTA are read
      // by quarters 0,1 (columns [0, N/2)) and again by 2,3 ([N/2, N))
      const int rq = ti.half ? (q & 1) * 32 : q * 32;
      // token-N tiling: the warp's 32 features (output columns) must exist
      // (the gate_up forward: the warp's 32 outputs)
      const bool warp_rows =
          C::SW ? (MODE == kFwdGateUp ? ti.n0 + crank * C::CH + (q & 1) * 32 < args.out[0].cols
                                      : ti.n0 + crank * 128 + q * 32 < args.out[0].cols)
                : C::kWgrad || ti.row0 + rq - __ldg(args.poff + ti.e) < __ldg(args.counts + ti.e);
      if (ti.active && warp_rows) {
        const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::ACC_COLS;
        const int row = ti.row0 + rq + lane;   // row-grouped modes: padded row of this thread
        const int orow = ti.row0 + rq;         // first row of this warp's output tiles
        float v[32];

        if constexpr (C::SW && MODE == kFwdGateUp) {
          // lane = feature, accumulator column = token of the unit.  Warps
          // q = 0, 1 hold the gate values of outputs o0 + lane, warps q + 2
          // the up values of the same outputs.  Per 32-token chunk each warp
          // saves its pre-activations, hands its partner the values of the
          // half of the tokens the partner finishes (gate warp: tokens
          // 16-31, up warp: 0-15), and applies the activation to its own
          // half.
          const bool up_w = q >= 2;
          const int o0 = ti.n0 + crank * C::CH + (q & 1) * 32;
          const int p0 = __ldg(args.poff + ti.e);
          const int left = min(__ldg(args.counts + ti.e) - (ti.row0 - p0), 256);   // tokens of the unit
          const int bar_id = 1 + (q & 1);
          float* mine = reinterpret_cast<float*>(my_epi);
          const float* peer = reinterpret_cast<const float*>(
              epi_g + ((warp - 2) ^ 2) * (C::EPI_WARP_BYTES + C::H1_WARP_BYTES));
          float b = 0.f;
          if (args.bias && o0 + lane < args.I)
            b = to_f32(static_cast<const T*>(args.bias)[static_cast<int64_t>(ti.e) * 2 * args.I +
                                                        (up_w ? args.I : 0) + o0 + lane]);
          auto run = [&](auto act_c) {
            constexpr int ACT = decltype(act_c)::value;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              if (c * 32 >= ti.nn) break;   // the same for both warps of the pair
              const int rows = left - c * 32;   // live tokens from this chunk on (>= 1)
              tmem_ld32(tacc + c * 32, v);
              if (args.bias) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] += b;
              }
              if (args.save_h1) {
                if (ACT == 1 && args.h1_half) {
                  // fp16 context (see h1_code_gate)
                  float hq[32];
#pragma unroll
                  for (int j = 0; j < 32; ++j)
                    hq[j] = up_w ? h1_code_up(v[j], args.limit) : h1_code_gate(v[j], args.limit);
                  store_tile_t16<__half, 32>(args.out[up_w ? 2 : 1], ti.row0 + c * 32, o0, hq, my_epi,
                                             lane, rows);
                } else {
                  store_tile_t(args.out[up_w ? 2 : 1], ti.row0 + c * 32, o0, v, my_epi, lane, rows,
                               [](int) { return 1.f; });
                }
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) mine[j * 32 + lane] = up_w ? v[j] : v[16 + j];
              pair_sync(bar_id);
              float a[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float o = peer[j * 32 + lane];
                a[j] = up_w ? act_fwd<ACT>(o, v[16 + j], args.limit, args.alpha)
                            : act_fwd<ACT>(v[j], o, args.limit, args.alpha);
              }
              pair_sync(bar_id);   // the partner has read this warp's half
              const int h0 = up_w ? 16 : 0;
              store_tile_t16<T, 16>(args.out[0], ti.row0 + c * 32 + h0, o0, a, my_epi, lane, rows - h0);
            }
          };
          if (args.act == 0)
            run(std::integral_constant<int, 0>{});
          else
            run(std::integral_constant<int, 1>{});
        } else if constexpr (C::SW) {
          // lane = feature (output column fcol + lane), accumulator column =
          // token of the unit: each 32-token chunk is transposed into token
          // rows; the down projection adds the bias and applies each token's
          // routing weight
          const int fcol = ti.n0 + crank * 128 + q * 32;
          const int p0 = __ldg(args.poff + ti.e);
          const int live = __ldg(args.counts + ti.e) - (ti.row0 - p0);   // tokens from row0
          const int g0 = __ldg(args.offsets + ti.e) + (ti.row0 - p0);
          float b = 0.f;
          if (MODE == kFwdDown && args.bias && fcol + lane < args.out[0].cols)
            b = to_f32(static_cast<const T*>(args.bias)[static_cast<int64_t>(ti.e) * args.out[0].cols + fcol + lane]);
          // routing weight of token 32 c + lane, for every chunk c, loaded up
          // front (independent loads); a row's weight then comes by shuffle
          float wt[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int tkn = c * 32 + lane;
            float wv = 0.f;
            if (MODE == kFwdDown && tkn < live && g0 + tkn < args.tk) {
              const int slot = __ldg(args.perm + g0 + tkn);
              if (slot >= 0 && slot < args.tk) wv = __ldg(args.topk_w + slot);
            }
            wt[c] = wv;
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            if (c * 32 >= ti.nn) break;   // warp-uniform
            tmem_ld32(tacc + c * 32, v);
            if (MODE == kFwdDown) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] += b;
            }
            const float wc = wt[c];
            store_tile_t(args.out[0], ti.row0 + c * 32, fcol, v, my_epi, lane,
                         min(32, live - c * 32), [&](int r) {
                           return MODE == kFwdDown ? __shfl_sync(0xffffffffu, wc, r) : 1.f;
                         });
          }
        } else if constexpr (C::kWgrad) {
          // fp32 weight gradients leave through TMA tensor stores: per 32-column
          // chunk, lane r writes row r's 128 bytes into a 32 x 32 staging tile
          // in the 128-byte swizzle (conflict-free 16-byte stores) and one lane
          // stores the tile; the staging tiles are used in turn.  Rows and
          // columns past the output are clipped by the store.
          if (ti.nkb > 0) {
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
              float w[32];
              tmem_ld32(tacc + c * 32, w);
              tma_store_tile32<C::STG_BUFS>(&maps.out, stg_buf(), w, ti.n0 + c * 32,
                                            ti.m0 + q * 32, ti.e, lane);
            }
          } else {
            // an expert without rows: every tile of the unit is zero, so one
            // zeroed staging tile feeds all of the warp's stores (one group)
            const uint32_t zb = stg_buf();
            if (lane == 0) bulk_wait_read<C::STG_BUFS - 1>();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) st_shared_v4(zb + lane * 128 + j * 16, 0.f, 0.f, 0.f, 0.f);
            fence_async_shared();
            __syncwarp();
            if (lane == 0) {
#pragma unroll 1
              for (int c = 0; c < BN / 32; ++c) tma_store_3d(&maps.out, zb, ti.n0 + c * 32, ti.m0 + q * 32, ti.e);
              bulk_commit();
            }
          }
        } else {
          // routing weight and liveness of this thread's row
          const int local = row - __ldg(args.poff + ti.e);
          const bool live = local < __ldg(args.counts + ti.e);
          float wrow = 0.f;
          if constexpr (MODE == kFwdDown || MODE == kDgradDown) {
            const int gi = __ldg(args.offsets + ti.e) + local;
            if (live && gi < args.tk) {
              const int slot = __ldg(args.perm + gi);
              if (slot >= 0 && slot < args.tk) wrow = __ldg(args.topk_w + slot);
            }
          }
          if constexpr (MODE == kFwdGateUp) {
            auto run = [&](auto act_c) {
            constexpr int ACT = decltype(act_c)::value;
            // output chunks of 32 columns; a half unit's warp takes the two
            // of its column half
            const int j0 = ti.half ? (q >> 1) * 2 : 0;
            const int j1 = ti.half ? j0 + 2 : BN / 64;
#pragma unroll 1
            for (int c = j0; c < j1; ++c) {
              // chunks past the last output column (the ragged last tile)
              // have nothing to compute
              if (ti.n0 + c * 32 >= args.I) break;
              float u[32];
              if constexpr (C::CTA2 && C::IL) {
                // 64 accumulator columns of gate/up pairs: gate at even, up
                // at odd columns
                const int pb = (ti.half ? 0 : (c >> 1) * 128) + (c & 1) * 64;
                float p0[32], p1[32];
                tmem_ld32(tacc + pb, p0);
                tmem_ld32(tacc + pb + 32, p1);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  v[i] = p0[2 * i];
                  u[i] = p0[2 * i + 1];
                  v[16 + i] = p1[2 * i];
                  u[16 + i] = p1[2 * i + 1];
                }
              } else {
                // (TF32, one CTA) accumulator columns [gate | up] of the tile
                static_assert(!C::CTA2, "pairs take interleaved columns here");
                tmem_ld32(tacc + c * 32, v);
                tmem_ld32(tacc + BN / 2 + c * 32, u);
              }
              if (args.bias) {
                // per-expert gate / up biases of this chunk's outputs
                const int i0 = ti.n0 + c * 32;
                const T* bg = static_cast<const T*>(args.bias) + static_cast<int64_t>(ti.e) * 2 * args.I;
                // interleaved bias columns also when the weights are read
                // through strided views (the fp32 path has no IL kernel)
                if (C::IL || args.gu_interleaved) {
                  float b[64];
#pragma unroll
                  for (int i = 0; i < 64; ++i) b[i] = 0.f;
                  add_bias(bg + 2 * i0, 2 * (args.I - i0), b);
#pragma unroll
                  for (int i = 0; i < 32; ++i) {
                    v[i] += b[2 * i];
                    u[i] += b[2 * i + 1];
                  }
                } else {
                  add_bias(bg + i0, args.I - i0, v);
                  add_bias(bg + args.I + i0, args.I - i0, u);
                }
              }
              if (args.save_h1) {
                if (ACT == 1 && !C::kTf32 && args.h1_half) {
                  // fp16 context (see h1_code_gate)
                  float gq[32], uq[32];
#pragma unroll
                  for (int i = 0; i < 32; ++i) {
                    gq[i] = h1_code_gate(v[i], args.limit);
                    uq[i] = h1_code_up(u[i], args.limit);
                  }
                  store_tile<__half>(args.out[1], 0, orow, ti.n0 + c * 32, gq, my_epi, lane);
                  store_tile<__half>(args.out[2], 0, orow, ti.n0 + c * 32, uq, my_epi, lane);
                } else {
                  store_tile<float>(args.out[1], 0, orow, ti.n0 + c * 32, v, my_epi, lane);
                  store_tile<float>(args.out[2], 0, orow, ti.n0 + c * 32, u, my_epi, lane);
                }
              }
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                v[i] = act_fwd<ACT>(v[i], u[i], args.limit, args.alpha);
                if constexpr (C::kTf32) v[i] = round_tf32(v[i]);   // operand of the down GEMM
              }
              store_tile<T>(args.out[0], 0, orow, ti.n0 + c * 32, v, my_epi, lane);
            }
            };
            if (args.act == 0)
              run(std::integral_constant<int, 0>{});
            else
              run(std::integral_constant<int, 1>{});
          } else if constexpr (MODE == kFwdDown || MODE == kDgradGateUp) {
            // fp32 rows for the combine; the down projection also applies the
            // routing weight of the row's slot
            const float scale = (MODE == kFwdDown) ? wrow : 1.f;
            // 64-column chunks; a half unit's warp takes those of its column
            // half, held in accumulator columns [0, N/2)
            const int c0 = ti.half ? (q >> 1) * (BN / 128) : 0;
            const int c1 = ti.half ? c0 + BN / 128 : BN / 64;
#pragma unroll 1
            for (int c = c0; c < c1; ++c) {
              if (ti.n0 + c * 64 >= args.out[0].cols) break;   // past the last output column
              float w2[64];
              tmem_ld64(tacc + (c - (ti.half ? c0 : 0)) * 64, w2);
              if (MODE == kFwdDown && args.bias) {
                // the expert's down bias, before the routing weight
                const int col = ti.n0 + c * 64;
                add_bias(static_cast<const T*>(args.bias) +
                             static_cast<int64_t>(ti.e) * args.out[0].cols + col,
                         args.out[0].cols - col, w2);
              }
#pragma unroll
              for (int i = 0; i < 64; ++i) w2[i] *= scale;
              store_tile<float>(args.out[0], 0, orow, ti.n0 + c * 64,
                                *reinterpret_cast<const float(*)[32]>(w2), my_epi, lane);
              store_tile<float>(args.out[0], 0, orow, ti.n0 + c * 64 + 32,
                                *reinterpret_cast<const float(*)[32]>(w2 + 32), my_epi, lane);
            }
          } else {  // kDgradDown
            // saved pre-activations of this row, gate at [0, I), up at [I, 2I):
            // fp32, or fp16 (h1_half, see h1_code_gate).  Each lane copies its
            // own row's 32 gate + 32 up values of a column chunk into shared
            // memory with cp.async, one chunk ahead.  A padding row reads
            // nothing: its staging is zero-filled (its dA' and routing weight
            // are zero, so its dH1 and w*a are zero whatever was saved).
            const int64_t h1off = static_cast<int64_t>(row) * 2 * args.I;   // elements
            const float* h1s = reinterpret_cast<const float*>(my_h1) + lane * 68;
            const uint32_t h1s_s = smem_u32(my_h1) + lane * 68 * 4;
            // column chunks that hold outputs (fewer in the ragged last tile)
            const int nch = min(BN / 32, (args.I - ti.n0 + 31) / 32);
            float dot = 0.f;
            auto run = [&](auto act_c) {
            constexpr int ACT = decltype(act_c)::value;
            // fp16 context: the clamped GLU only (the host sets h1_half)
            const bool half = (ACT == 1 && !C::kTf32 && args.h1_half);
            // I % 8 == 0: 16-byte units are all inside the row or all past it
            auto prefetch = [&](int c) {
              const int i0 = ti.n0 + c * 32;
              if (half) {
                const __half* h1row = static_cast<const __half*>(args.h1) + h1off;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const int col = i0 + 8 * j;
                  const bool in = live && col < args.I;
                  cp_async16(h1s_s + j * 16, in ? h1row + col : h1row, in ? 16u : 0u);
                  cp_async16(h1s_s + 64 + j * 16, in ? h1row + args.I + col : h1row, in ? 16u : 0u);
                }
              } else {
                const float* h1row = static_cast<const float*>(args.h1) + h1off;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const int col = i0 + 4 * j;
                  const bool in = live && col < args.I;
                  cp_async16(h1s_s + j * 16, in ? h1row + col : h1row, in ? 16u : 0u);
                  cp_async16(h1s_s + 128 + j * 16, in ? h1row + args.I + col : h1row, in ? 16u : 0u);
                }
              }
              cp_async_commit();
            };
            prefetch(0);
#pragma unroll 1
            for (int c = 0; c < nch; ++c) {
              tmem_ld32(tacc + c * 32, v);   // dA' (before the routing weight)
              const int i0 = ti.n0 + c * 32;
              float g[32], u[32];
              cp_async_wait_all();
              if (half) {
                const uint4* hs = reinterpret_cast<const uint4*>(h1s);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const uint4 gv = hs[j], uv = hs[4 + j];
                  const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    const float2 gf = __half22float2(*reinterpret_cast<const __half2*>(&gw[i]));
                    const float2 uf = __half22float2(*reinterpret_cast<const __half2*>(&uw[i]));
                    g[8 * j + 2 * i] = gf.x; g[8 * j + 2 * i + 1] = gf.y;
                    u[8 * j + 2 * i] = uf.x; u[8 * j + 2 * i + 1] = uf.y;
                  }
                }
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float4 gv = *reinterpret_cast<const float4*>(h1s + 4 * j);
                  const float4 uv = *reinterpret_cast<const float4*>(h1s + 32 + 4 * j);
                  g[4 * j] = gv.x; g[4 * j + 1] = gv.y; g[4 * j + 2] = gv.z; g[4 * j + 3] = gv.w;
                  u[4 * j] = uv.x; u[4 * j + 1] = uv.y; u[4 * j + 2] = uv.z; u[4 * j + 3] = uv.w;
                }
              }
              // refill the staging row with the next chunk as early as possible:
              // a use of every value read above orders those reads before the
              // copies that overwrite them
              if (c + 1 < nch) {
                float any = 0.f;
#pragma unroll
                for (int i = 0; i < 32; ++i) any += g[i] + u[i];
                asm volatile("" ::"f"(any));
                prefetch(c + 1);
              }
              float dg[32], du[32], aw[32];
              // two elements per step on the packed fp32 pipe; the dot
              // product keeps an even and an odd partial sum
              const float2 w2 = make_float2(wrow, wrow);
              float2 dot2 = make_float2(0.f, 0.f);
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                float2 a, pg, pu;
                act_bwd2<ACT>(make_float2(g[i], g[i + 1]), make_float2(u[i], u[i + 1]),
                              args.limit, args.alpha, a, pg, pu);
                const float2 vv = make_float2(v[i], v[i + 1]);
                dot2 = __ffma2_rn(vv, a, dot2);
                const float2 da = __fmul2_rn(w2, vv);
                const float2 rg = __fmul2_rn(da, pg), ru = __fmul2_rn(da, pu), ra = __fmul2_rn(w2, a);
                dg[i] = rg.x; dg[i + 1] = rg.y;
                du[i] = ru.x; du[i + 1] = ru.y;
                aw[i] = ra.x; aw[i + 1] = ra.y;
              }
              dot += dot2.x + dot2.y;
              if constexpr (C::kTf32) {
                // operands of the TF32 dgrad / wgrad products
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  dg[i] = round_tf32(dg[i]);
                  du[i] = round_tf32(du[i]);
                  aw[i] = round_tf32(aw[i]);
                }
                if constexpr (C::IL) {
                  // dgate / dup of output i are columns 2i, 2i + 1 of dH1
#pragma unroll
                  for (int hh = 0; hh < 2; ++hh) {
                    float t[32];
#pragma unroll
                    for (int p = 0; p < 16; ++p) {
                      t[2 * p] = dg[16 * hh + p];
                      t[2 * p + 1] = du[16 * hh + p];
                    }
                    store_tile<T>(args.out[0], 0, orow, 2 * i0 + 32 * hh, t, my_epi, lane);
                  }
                } else {
                  store_tile<T>(args.out[0], 0, orow, i0, dg, my_epi, lane);
                  store_tile<T>(args.out[1], 0, orow, i0, du, my_epi, lane);
                }
                store_tile<T>(args.out[2], 0, orow, i0, aw, my_epi, lane);
              } else if constexpr (C::IL) {
                // dgate / dup of output i are columns 2i, 2i + 1 of dH1: bf16
                // hi parts, then (for experts that need them) the remainders,
                // of 16 outputs at a time
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  float t[32];
#pragma unroll
                  for (int p = 0; p < 16; ++p) {
                    t[2 * p] = bf16_round(dg[16 * hh + p]);
                    t[2 * p + 1] = bf16_round(du[16 * hh + p]);
                  }
                  store_tile<T>(args.out[0], 0, orow, 2 * i0 + 32 * hh, t, my_epi, lane);
                  if (ti.lo) {
#pragma unroll
                    for (int p = 0; p < 16; ++p) {
                      t[2 * p] = dg[16 * hh + p] - bf16_round(dg[16 * hh + p]);
                      t[2 * p + 1] = du[16 * hh + p] - bf16_round(du[16 * hh + p]);
                    }
                    store_tile<T>(args.out[3], 0, orow, 2 * i0 + 32 * hh, t, my_epi, lane);
                  }
                }
                if (ti.lo) {
                  float lo[32];
#pragma unroll
                  for (int i = 0; i < 32; ++i) split_bf16(aw[i], aw[i], lo[i]);
                  store_tile<T>(args.out[5], 0, orow, i0, lo, my_epi, lane);
                }
                store_tile<T>(args.out[2], 0, orow, i0, aw, my_epi, lane);
              } else if (!ti.lo) {
                // one bf16 value per operand (the store rounds to nearest)
                store_tile<T>(args.out[0], 0, orow, i0, dg, my_epi, lane);
                store_tile<T>(args.out[1], 0, orow, i0, du, my_epi, lane);
                store_tile<T>(args.out[2], 0, orow, i0, aw, my_epi, lane);
              } else {
                // bf16 hi parts (operands of the dgrad and the wgrads) and lo
                // parts (the remainders, operands of the wgrads only)
                float lo[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) split_bf16(dg[i], dg[i], lo[i]);
                store_tile<T>(args.out[0], 0, orow, i0, dg, my_epi, lane);
                store_tile<T>(args.out[3], 0, orow, i0, lo, my_epi, lane);
#pragma unroll
                for (int i = 0; i < 32; ++i) split_bf16(du[i], du[i], lo[i]);
                store_tile<T>(args.out[1], 0, orow, i0, du, my_epi, lane);
                store_tile<T>(args.out[4], 0, orow, i0, lo, my_epi, lane);
#pragma unroll
                for (int i = 0; i < 32; ++i) split_bf16(aw[i], aw[i], lo[i]);
                store_tile<T>(args.out[2], 0, orow, i0, aw, my_epi, lane);
                store_tile<T>(args.out[5], 0, orow, i0, lo, my_epi, lane);
              }
            }
            };
            if (args.act == 0)
              run(std::integral_constant<int, 0>{});
            else
              run(std::integral_constant<int, 1>{});
            args.dwpart[static_cast<int64_t>(ti.nt) * args.rows_max + row] = live ? dot : 0.f;
          }
        }
      }
      // release the accumulator to the MMA issuer (the leader): every lane's
      // tensor-memory reads have completed (tcgen05.wait::ld) and are fenced
      // before the warp's single arrival.  The arrival orders nothing else:
      // the odd CTA's remote arrival is relaxed, since a cluster-scope
      // release would first drain all of the warp's global stores.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (C::CTA2 && !leader)
          mbar_arrive_cluster_relaxed(leader_addr(tempty_bar + 8 * acc));
        else
          mbar_arrive(tempty_bar + 8 * acc);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // the weight gradients' tensor stores must be complete before the CTA exits
    if constexpr (C::TMA_OUT) {
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  // Every MMA of the pair has completed once the drain barrier has seen the
  // leader's final commit; only then may tensor memory be freed and the CTAs
  // exit (the cluster barrier also keeps each CTA alive while its peer may
  // still signal its barriers).
  if (warp == 1 && lane == 0 && !mbar_wait(drain_bar, 0, kDrainNs))
    record_error(args.err, kErrTimeout);
  __syncthreads();
  if constexpr (C::CTA2) cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (C::CTA2)
      tmem_dealloc2(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <typename T, int MODE, int BN, int STAGES, bool IL = false, bool SW = false>
cudaError_t launch_gemm_t(const GemmMaps& maps, const GemmArgs& args, int num_sms,
                          cudaStream_t st) {
  using C = GemmCfg<T, MODE, BN, STAGES, IL, SW>;
  auto kern = moe_gemm_kernel<T, MODE, BN, STAGES, IL, SW>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool configured[64] = {};
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms / C::PAIR * C::PAIR));
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C::PAIR;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps, args);
}

}  // namespace moe
