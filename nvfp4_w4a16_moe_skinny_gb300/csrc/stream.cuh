// Per-warp weight streaming, the chunk consumers and activation staging (sm_103a).
//
// A *chunk* is the tiles of one 64-row group and one 64-column slice of K (four
// 576-byte tiles, 2,304 contiguous bytes in the repacked layout, version 2).  A
// warp streams 1 to 4 adjacent tiles of a group through its private ring of
// `ns` 2,304-byte stages in shared memory.  Lane 0 fills a stage with one tiled
// tensor copy (TMA engine, L2 evict-first) of those tiles over 1, 2 or 4
// consecutive chunks (4 tiles x 1, 3 x 1, 2 x 2 or 1 x 4 chunks); the whole warp
// waits on the stage's mbarrier; when the warp has consumed a stage, lane 0
// refills it with the copy `ns` positions ahead.  No stage is shared between
// warps, so the only synchronisation is the mbarrier (copy -> warp) and
// __syncwarp (warp -> refill).
//
// Activations are staged once per CTA as f16 rows (each row rescaled by a power
// of two), 128 bytes per row and 64-column chunk, one warp per row.  A consumer
// reaches the rows of its token slots through per-lane row addresses, so one
// staged copy of the tokens serves every expert of a grouped product.
//
// Chunk consumers:
//  * mma_chunk<NT, TN>: tensor cores (m16n8k16, f16 in, f32 accumulate); each
//    tile's 16 rows are the A operand and up to 8*NT token slots the N operand.
//    The x fragments of the 64 columns are loaded once and feed the TN tiles.
//    Each E2M1 pair goes through the hardware converter and is multiplied in f16
//    by its E4M3 scale (exact: the product has at most 6 significant bits).
//  * core_chunk<TN>: CUDA cores for one token.  Lane (g, q) takes rows g and
//    g+8 of each tile over the 16-column group q; it sums E2M1 x activation
//    products in f32 (mixed-precision FMA; the products are exact) and scales
//    each group sum once.  The cross-lane sum over q is left to warp shuffles in
//    the epilogue.  (Two or more tokens run on an 8-slot tensor-core column:
//    one FMA per weight and token cost more than the MMA from two tokens up.)
#pragma once

#include "common.cuh"

namespace nvfp4 {

constexpr int kChunkTiles = 4;                          // tiles per chunk (one 64-row group)
constexpr int kStageBytes = kChunkTiles * kTileBytes;   // 2,304 bytes
// Staged activations: bytes per row and 64-column chunk (32 f16 pairs).  MMA
// order: lane (g, t) reads 32 contiguous bytes at 32*t, word 2*kt + h holding
// columns 16*kt + 2*t + 8*h (+1) -- the m16n8k16 B fragment of token slot g.
// CUDA-core order: pair j (columns 2j, 2j+1) at word j.
constexpr int kXChunkBytes = 128;

template <int NT>
__device__ __forceinline__ void mma_step(uint32_t word, uint32_t s, const uint32_t (&b0)[NT],
                                         const uint32_t (&b1)[NT], float (&acc)[NT][4]) {
  uint32_t h[4];
  e2m1x8_to_f16x2(word, h);
  uint32_t a[4];
  hmul2_bcast(h[0], h[1], s, a[0], a[1]);  // rows g, g+8, columns 2t, 2t+1
  hmul2_bcast(h[2], h[3], s, a[2], a[3]);  // rows g, g+8, columns 2t+8, 2t+9
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) mma_f16(acc[nt], a, b0[nt], b1[nt]);
}

// TN tiles at shared address `st` against x fragments at xr[nt] (this lane's 32
// bytes of slot 8*nt + g for the chunk).  acc[r][nt] is tile r's C fragment:
// [0],[1] = row g, slots 8nt+2t, +1; [2],[3] = row g+8.
template <int NT, int TN, int NR>
__device__ __forceinline__ void mma_chunk(uint32_t st, const uint32_t (&xr)[NT], int lane,
                                          float (&acc)[NR][NT][4]) {
  static_assert(TN <= NR, "one accumulator per tile");
  uint4 xa[NT], xb[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    xa[nt] = lds128(xr[nt]);
    xb[nt] = lds128(xr[nt] + 16);
  }
  uint4 wv[TN];
  uint2 sv[TN];
#pragma unroll
  for (int r = 0; r < TN; ++r) {
    wv[r] = lds128(st + r * kTileBytes + lane * 16);
    sv[r] = lds64(st + r * kTileBytes + kTileNibBytes + (lane >> 2) * 8);
  }
  uint32_t b0[NT], b1[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) b0[nt] = xa[nt].x, b1[nt] = xa[nt].y;
#pragma unroll
  for (int r = 0; r < TN; ++r) mma_step<NT>(wv[r].x, scale_pair_lohi<0, 1>(sv[r].x), b0, b1, acc[r]);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) b0[nt] = xa[nt].z, b1[nt] = xa[nt].w;
#pragma unroll
  for (int r = 0; r < TN; ++r) mma_step<NT>(wv[r].y, scale_pair_lohi<2, 3>(sv[r].x), b0, b1, acc[r]);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) b0[nt] = xb[nt].x, b1[nt] = xb[nt].y;
#pragma unroll
  for (int r = 0; r < TN; ++r) mma_step<NT>(wv[r].z, scale_pair_lohi<0, 1>(sv[r].y), b0, b1, acc[r]);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) b0[nt] = xb[nt].z, b1[nt] = xb[nt].w;
#pragma unroll
  for (int r = 0; r < TN; ++r) mma_step<NT>(wv[r].w, scale_pair_lohi<2, 3>(sv[r].y), b0, b1, acc[r]);
}

// Per-lane constants of the CUDA-core consumer: lane (g, q) reads, at step j, the
// 32-bit word q of lane-chunk t_j = (j + g/2) & 3 of row pair g (the rotation by
// g/2 puts the 32 lanes on 32 distinct banks) and the x pairs 8q + t_j, 8q + t_j + 4.
struct CoreLane {
  uint32_t w_off[4];  // byte offset of the weight word within a tile
  uint32_t x_off[4];  // byte offset of x pair 8q + t_j within a row's 64-column chunk
  uint32_t s_off;     // byte offset of the scale pair (rows g, g+8; group q) within a tile
  __device__ __forceinline__ CoreLane(int lane) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = (j + (g >> 1)) & 3;
      w_off[j] = 16 * (4 * g + t) + 4 * q;
      x_off[j] = (8 * q + t) * 4;
    }
    s_off = kTileNibBytes + 8 * g + 2 * q;
  }
};

// TN tiles at `st` on CUDA cores for one token (MT == 1).  xr[0]: the token's
// staged row for this chunk.  acc[r][0][0] = tile r, row g; acc[r][0][1] = row
// g+8 (partial over group q).
template <int MT, int TN>
__device__ __forceinline__ void core_chunk(uint32_t st, const uint32_t (&xr)[MT], const CoreLane& cl,
                                           float (&acc)[4][MT][2]) {
  static_assert(MT == 1, "the CUDA-core consumer serves one token");
  uint32_t xw[4][2];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    xw[j][0] = lds32(xr[0] + cl.x_off[j]);
    xw[j][1] = lds32(xr[0] + cl.x_off[j] + 16);
  }
#pragma unroll
  for (int r = 0; r < TN; ++r) {
    const uint32_t tile = st + r * kTileBytes;
    const uint32_t sp = scale_pair_lohi<0, 1>(lds16(tile + cl.s_off));
    float pa = 0.f, pb = 0.f, pc = 0.f, pd = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t hh[4];
      e2m1x8_to_f16x2(lds32(tile + cl.w_off[j]), hh);
      pa = fma_f16lo(hh[0], xw[j][0], pa);
      pb = fma_f16hi(hh[0], xw[j][0], pb);
      pa = fma_f16lo(hh[2], xw[j][1], pa);
      pb = fma_f16hi(hh[2], xw[j][1], pb);
      pc = fma_f16lo(hh[1], xw[j][0], pc);
      pd = fma_f16hi(hh[1], xw[j][0], pd);
      pc = fma_f16lo(hh[3], xw[j][1], pc);
      pd = fma_f16hi(hh[3], xw[j][1], pd);
    }
    const float sg = f16lo_to_f32(sp), sg8 = f16hi_to_f32(sp);  // scale * 2^-8
    acc[r][0][0] = fmaf(pa + pb, sg, acc[r][0][0]);
    acc[r][0][1] = fmaf(pc + pd, sg8, acc[r][0][1]);
  }
}

// Chunks per copy for a piece of tn tiles: a copy (one TMA box) carries tn tiles
// of copy_chunks(tn) consecutive chunks, at most kStageBytes.
__host__ __device__ constexpr int copy_chunks(int tn) { return tn == 1 ? 4 : (tn == 2 ? 2 : 1); }

// The TMA view of a repacked weight (stack): a 4-D tensor of 8-byte elements,
// dims (72 = one tile's 576 bytes, 4 tiles of a chunk, kc chunks, groups of
// all matrices), so the box (72, tn, copy_chunks(tn), 1) at (0, t0, c, group)
// is tiles t0..t0+tn-1 of chunks c, c+1, ... of one group, stored in shared
// memory chunk-major: [chunk][tile][576 bytes].
struct WeightMaps {
  CUtensorMap w[4];   // the (stacked) weight; w[tn - 1] has the box of tn tiles
  CUtensorMap sh[4];  // the shared expert of a MoE layer (unused otherwise)
};

// The f16 pairs h[0..3] of columns 8*c8 .. 8*c8+7 (pair e = columns 2e, 2e+1,
// low half first) of a staged row at rowp: the m16n8k16 B-fragment order (MMA)
// or pair order (CUDA cores) of their 64-column chunk.
template <bool kMMA>
__device__ __forceinline__ void place8(uint8_t* rowp, int c8, const uint32_t (&h)[4]) {
  const int kcl = c8 >> 3, c64 = (c8 & 7) * 8;  // chunk, first column within the chunk
  uint8_t* cp = rowp + kcl * kXChunkBytes;
  if constexpr (kMMA) {
    // columns c64..c64+7 = k-step kt, half hf, pairs t = 0..3 -> word 8t + 2kt + hf
    uint32_t* dst = reinterpret_cast<uint32_t*>(cp) + (c64 >> 4) * 2 + ((c64 >> 3) & 1);
#pragma unroll
    for (int t = 0; t < 4; ++t) dst[t * 8] = h[t];
  } else {
    *reinterpret_cast<uint4*>(cp + c64 * 2) = make_uint4(h[0], h[1], h[2], h[3]);
  }
}

// Stage `nrows` bf16 rows of x (row_src[j] = source row, row length k) over
// columns [col0, col0 + 64*nchunks) into shared memory as f16, row j rescaled by
// 2^sigma[j] (sigma from the row's amax over the same columns, see
// pow2_rescale_exponent), followed by one all-zero row (index nrows) that empty
// token slots point at.  Row j starts at xs + j*stride.  One warp per row: the
// lanes load the row's 16-byte groups (8 columns each), take the amax with warp
// shuffles, then convert and store in the MMA fragment order or the CUDA-core
// pair order.  Rows of up to 32*kStageRegs groups are read once and held in
// registers; longer rows are read twice.  Columns at or past k are stored as
// zeros.  `after_loads` runs in each warp once its first row's loads are issued
// (the caller issues the rest of its weight copies behind them; it must be safe
// to call again).  All threads of the CTA call it; it ends with a __syncthreads.
constexpr int kStageRegs = 12;

template <bool kMMA, typename F>
__device__ __forceinline__ void stage_rows(const uint16_t* __restrict__ x, int k, int col0, int nchunks, int nrows,
                                           const int* row_src, int* sigma, uint8_t* xs, int stride, F&& after_loads) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int groups = nchunks * 8;  // 8-column groups per row
  const bool one_pass = groups <= 32 * kStageRegs;
  auto amax8 = [](const uint4& v) {
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    float am = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      am = fmaxf(am, fmaxf(fabsf(__uint_as_float(w4[e] << 16)), fabsf(__uint_as_float(w4[e] & 0xFFFF0000u))));
    return am;
  };
  auto store8 = [&](uint8_t* rowp, int c8, const uint4& v, float sc) {
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(w4[e] << 16) * sc, hi = __uint_as_float(w4[e] & 0xFFFF0000u) * sc;
      h[e] = f32x2_to_f16x2(lo, hi);
    }
    place8<kMMA>(rowp, c8, h);
  };
  for (int row = warp; row <= nrows; row += nwarps) {
    uint8_t* rowp = xs + static_cast<size_t>(row) * stride;
    if (row == nrows) {  // the zero row
      for (int b = lane * 16; b < nchunks * kXChunkBytes; b += 32 * 16) *reinterpret_cast<uint4*>(rowp + b) = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint16_t* src = x + static_cast<size_t>(row_src[row]) * k + col0;
    const int lim = k - col0;  // columns of this row that exist
    auto load8 = [&](int c8) -> uint4 {
      return (c8 < groups && c8 * 8 < lim) ? __ldg(reinterpret_cast<const uint4*>(src + c8 * 8)) : make_uint4(0, 0, 0, 0);
    };
    uint4 v[kStageRegs];
    float am = 0.f;
    if (one_pass) {
#pragma unroll
      for (int j = 0; j < kStageRegs; ++j) v[j] = load8(lane + 32 * j);
      after_loads();
#pragma unroll
      for (int j = 0; j < kStageRegs; ++j) am = fmaxf(am, amax8(v[j]));
    } else {
      for (int b = 0; b < groups; b += 32 * kStageRegs) {
#pragma unroll
        for (int j = 0; j < kStageRegs; ++j) v[j] = load8(b + lane + 32 * j);
        if (b == 0) after_loads();
#pragma unroll
        for (int j = 0; j < kStageRegs; ++j) am = fmaxf(am, amax8(v[j]));
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
    const int sg = pow2_rescale_exponent(am);
    if (lane == 0) sigma[row] = sg;
    const float sc = exp2i(sg);
    if (one_pass) {
#pragma unroll
      for (int j = 0; j < kStageRegs; ++j)
        if (lane + 32 * j < groups) store8(rowp, lane + 32 * j, v[j], sc);
    } else {
      for (int b = 0; b < groups; b += 32 * kStageRegs) {
#pragma unroll
        for (int j = 0; j < kStageRegs; ++j) v[j] = load8(b + lane + 32 * j);
#pragma unroll
        for (int j = 0; j < kStageRegs; ++j)
          if (b + lane + 32 * j < groups) store8(rowp, b + lane + 32 * j, v[j], sc);
      }
    }
  }
  after_loads();
  __syncthreads();
}

// The same staging for activations already quantized to NVFP4 (the W4A4
// products): canonical codes [rows, k/2] and E4M3 scales [rows, k/16] of row
// row_src[j], each 16-column group dequantized as e2m1 * e4m3 * 2^-8 in f16 --
// exact, as for the weights (at most 6 significant bits, within f16's range) --
// and sigma[j] = -8, so that the epilogue's 2^(8 - sigma) restores the 2^-8;
// the row's global scale is applied by the caller's multiplier.
template <bool kMMA, typename F>
__device__ __forceinline__ void stage_rows_fp4(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scl,
                                               int k, int col0, int nchunks, int nrows, const int* row_src,
                                               int* sigma, uint8_t* xs, int stride, F&& after_loads) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int groups = nchunks * 8;  // 8-column groups per row
  after_loads();  // the rows are read once, with nothing to overlap: issue the copies first
  for (int row = warp; row <= nrows; row += nwarps) {
    uint8_t* rowp = xs + static_cast<size_t>(row) * stride;
    if (row == nrows) {  // the zero row
      for (int b = lane * 16; b < nchunks * kXChunkBytes; b += 32 * 16) *reinterpret_cast<uint4*>(rowp + b) = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint8_t* crow = codes + static_cast<size_t>(row_src[row]) * (k / 2) + col0 / 2;
    const uint8_t* srow = scl + static_cast<size_t>(row_src[row]) * (k / 16) + col0 / 16;
    const int lim = k - col0;  // columns of this row that exist
    for (int c8 = lane; c8 < groups; c8 += 32) {
      uint32_t h[4] = {0u, 0u, 0u, 0u};
      if (c8 * 8 < lim) {
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(crow + c8 * 4));
        const uint32_t sb = __ldg(srow + (c8 >> 1));
        e2m1x8_to_f16x2(w, h);
        const uint32_t s2 = scale_pair_lohi<0, 0>(sb);  // [e4m3, e4m3] * 2^-8
#pragma unroll
        for (int e = 0; e < 4; ++e) h[e] = hmul2(h[e], s2);
      }
      place8<kMMA>(rowp, c8, h);
    }
    if (lane == 0) sigma[row] = -8;
  }
  __syncthreads();
}

}  // namespace nvfp4
