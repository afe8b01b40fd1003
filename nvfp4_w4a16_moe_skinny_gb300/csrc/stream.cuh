// Per-warp weight streaming and the chunk consumers (sm_103a).
//
// A *chunk* is the four 576-byte tiles of one 64-row group and one 64-column
// slice of K (2,304 contiguous bytes in the repacked layout, version 2).  Every
// warp owns a private ring of `ns` chunk-sized stages in shared memory.  Lane 0
// fills a stage with one 1-D bulk copy (TMA engine, L2 evict-first); the whole
// warp waits on the stage's mbarrier; when the warp has consumed a stage, lane 0
// refills it with the chunk `ns` positions ahead.  No stage is shared between
// warps, so the only synchronisation is the mbarrier (copy -> warp) and
// __syncwarp (warp -> refill).
//
// Chunk consumers:
//  * mma_chunk<NT>: tensor cores (m16n8k16, f16 in, f32 accumulate); each tile's
//    16 rows are the A operand and up to 8*NT tokens the N operand.  The x
//    fragments of the 64 columns are loaded once and feed the four tiles, which
//    also gives four independent accumulator chains.  Each E2M1 pair goes
//    through the hardware converter and is multiplied in f16 by its E4M3 scale
//    (exact: the product has at most 6 significant bits).
//  * core_chunk<MT>: CUDA cores for up to 7 tokens.  Lane (g, q) takes rows g and
//    g+8 of each tile over the 16-column group q; it sums E2M1 x activation
//    products in f32 (mixed-precision FMA; the products are exact) and scales
//    each group sum once (MT <= 2), or scales the weights in f16 first and
//    accumulates directly (MT >= 3, fewer live registers).  The cross-lane sum
//    over q is left to warp shuffles in the epilogue.
#pragma once

#include "common.cuh"

namespace nvfp4 {

constexpr int kChunkTiles = 4;                          // tiles per chunk (one 64-row group)
constexpr int kStageBytes = kChunkTiles * kTileBytes;   // 2,304 bytes

// x fragments for the MMA path, per 64-column chunk and 8-token group: 32 lanes x
// 8 words (f16x2).  Lane (g, t), word 2*kt + h holds token slot g, columns
// 16*kt + 2*t + 8*h (+1) of the chunk -- the m16n8k16 B fragment.
constexpr int kXFragChunkBytes = 1024;
// x for the CUDA-core path, per 64-column chunk and token: 32 f16x2 words (pairs).
constexpr int kXCoreChunkBytes = 128;

template <int NT>
__device__ __forceinline__ void mma_step(uint32_t word, uint32_t sg, uint32_t sg8, const uint32_t (&b0)[NT],
                                         const uint32_t (&b1)[NT], float (&acc)[NT][4]) {
  uint32_t h[4];
  e2m1x8_to_f16x2(word, h);
  uint32_t a[4];
  a[0] = hmul2(h[0], sg);   // row g,   columns 2t, 2t+1
  a[1] = hmul2(h[1], sg8);  // row g+8, columns 2t, 2t+1
  a[2] = hmul2(h[2], sg);   // row g,   columns 2t+8, 2t+9
  a[3] = hmul2(h[3], sg8);  // row g+8, columns 2t+8, 2t+9
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) mma_f16(acc[nt], a, b0[nt], b1[nt]);
}

// One chunk (4 tiles at `st`) against x fragments `xf` (NT * 1024 bytes).
// acc[r][nt] is tile r's C fragment: [0],[1] = row g, tokens 8nt+2t, +1; [2],[3] = row g+8.
template <int NT>
__device__ __forceinline__ void mma_chunk(const uint8_t* st, const uint8_t* xf, int lane, float (&acc)[4][NT][4]) {
  uint4 xa[NT], xb[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    xa[nt] = lds128(xf + nt * kXFragChunkBytes + lane * 32);
    xb[nt] = lds128(xf + nt * kXFragChunkBytes + lane * 32 + 16);
  }
  uint4 wv[4];
  uint2 sv[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    wv[r] = lds128(st + r * kTileBytes + lane * 16);
    sv[r] = lds64(st + r * kTileBytes + kTileNibBytes + (lane >> 2) * 8);
  }
  uint32_t b0[NT], b1[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) b0[nt] = xa[nt].x, b1[nt] = xa[nt].y;
#pragma unroll
  for (int r = 0; r < 4; ++r) mma_step<NT>(wv[r].x, scale_pair_x2<0>(sv[r].x), scale_pair_x2<1>(sv[r].x), b0, b1, acc[r]);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) b0[nt] = xa[nt].z, b1[nt] = xa[nt].w;
#pragma unroll
  for (int r = 0; r < 4; ++r) mma_step<NT>(wv[r].y, scale_pair_x2<2>(sv[r].x), scale_pair_x2<3>(sv[r].x), b0, b1, acc[r]);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) b0[nt] = xb[nt].x, b1[nt] = xb[nt].y;
#pragma unroll
  for (int r = 0; r < 4; ++r) mma_step<NT>(wv[r].z, scale_pair_x2<0>(sv[r].y), scale_pair_x2<1>(sv[r].y), b0, b1, acc[r]);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) b0[nt] = xb[nt].z, b1[nt] = xb[nt].w;
#pragma unroll
  for (int r = 0; r < 4; ++r) mma_step<NT>(wv[r].w, scale_pair_x2<2>(sv[r].y), scale_pair_x2<3>(sv[r].y), b0, b1, acc[r]);
}

__device__ __forceinline__ uint32_t lds_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(smem_addr(p)));
  return v;
}

// Per-lane constants of the CUDA-core consumer: lane (g, q) reads, at step j, the
// 32-bit word q of lane-chunk t_j = (j + g/2) & 3 of row pair g (the rotation by
// g/2 puts the 32 lanes on 32 distinct banks) and the x pairs 8q + t_j, 8q + t_j + 4.
struct CoreLane {
  int w_off[4];   // byte offset of the weight word within a tile
  int x_off[4];   // byte offset of x pair 8q + t_j within a token's 64-column chunk
  int s_off;      // byte offset of the scale pair (rows g, g+8; group q) within a tile
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

// One chunk on CUDA cores.  xw: the chunk's x words [MT][32 words].  acc[r][m][0]
// = tile r, row g; acc[r][m][1] = row g+8 (partial over this lane's group q).
template <int MT>
__device__ __forceinline__ void core_chunk(const uint8_t* st, const uint8_t* xw, const CoreLane& cl,
                                           float (&acc)[4][MT][2]) {
  if constexpr (MT <= 2) {
    uint32_t xr[MT][4][2];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        xr[m][j][0] = lds32(xw + m * kXCoreChunkBytes + cl.x_off[j]);
        xr[m][j][1] = lds32(xw + m * kXCoreChunkBytes + cl.x_off[j] + 16);
      }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint8_t* tile = st + r * kTileBytes;
      const uint32_t sp = scale_lohi_x2(lds_u16(tile + cl.s_off));
      float pa[MT], pb[MT], pc[MT], pd[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) pa[m] = pb[m] = pc[m] = pd[m] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t hh[4];
        e2m1x8_to_f16x2(lds32(tile + cl.w_off[j]), hh);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          pa[m] = fma_f16lo(hh[0], xr[m][j][0], pa[m]);
          pb[m] = fma_f16hi(hh[0], xr[m][j][0], pb[m]);
          pa[m] = fma_f16lo(hh[2], xr[m][j][1], pa[m]);
          pb[m] = fma_f16hi(hh[2], xr[m][j][1], pb[m]);
          pc[m] = fma_f16lo(hh[1], xr[m][j][0], pc[m]);
          pd[m] = fma_f16hi(hh[1], xr[m][j][0], pd[m]);
          pc[m] = fma_f16lo(hh[3], xr[m][j][1], pc[m]);
          pd[m] = fma_f16hi(hh[3], xr[m][j][1], pd[m]);
        }
      }
      const float sg = f16lo_to_f32(sp), sg8 = f16hi_to_f32(sp);  // scale * 2^-8
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        acc[r][m][0] = fmaf(pa[m] + pb[m], sg, acc[r][m][0]);
        acc[r][m][1] = fmaf(pc[m] + pd[m], sg8, acc[r][m][1]);
      }
    }
  } else {
    uint32_t sgd[4], sg8d[4];  // (scale, scale) * 2^-8 per tile for rows g and g+8
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint32_t sw = lds_u16(st + r * kTileBytes + cl.s_off);
      sgd[r] = scale_pair_x2<0>(sw);
      sg8d[r] = scale_pair_x2<1>(sw);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t x0[MT], x1[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        x0[m] = lds32(xw + m * kXCoreChunkBytes + cl.x_off[j]);
        x1[m] = lds32(xw + m * kXCoreChunkBytes + cl.x_off[j] + 16);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        uint32_t hh[4];
        e2m1x8_to_f16x2(lds32(st + r * kTileBytes + cl.w_off[j]), hh);
        const uint32_t h0 = hmul2(hh[0], sgd[r]), h2 = hmul2(hh[2], sgd[r]);
        const uint32_t h1 = hmul2(hh[1], sg8d[r]), h3 = hmul2(hh[3], sg8d[r]);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          float a0 = acc[r][m][0], a1 = acc[r][m][1];
          a0 = fma_f16lo(h0, x0[m], a0);
          a0 = fma_f16hi(h0, x0[m], a0);
          a0 = fma_f16lo(h2, x1[m], a0);
          a0 = fma_f16hi(h2, x1[m], a0);
          a1 = fma_f16lo(h1, x0[m], a1);
          a1 = fma_f16hi(h1, x0[m], a1);
          a1 = fma_f16lo(h3, x1[m], a1);
          a1 = fma_f16hi(h3, x1[m], a1);
          acc[r][m][0] = a0, acc[r][m][1] = a1;
        }
      }
    }
  }
}

// Shared-memory ring of one warp.
struct Ring {
  uint8_t* buf;    // ns * kStageBytes
  uint64_t* bar;   // ns mbarriers
  int ns;
};

__device__ __forceinline__ void ring_init(const Ring& r, int lane) {
  if (lane == 0) {
    for (int s = 0; s < r.ns; ++s) mbar_init(&r.bar[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
}

// Lane 0 only: copy the chunk at `src` (kStageBytes) into stage s.
__device__ __forceinline__ void ring_issue(const Ring& r, int s, const uint8_t* src, uint64_t policy) {
  mbar_arrive_expect_tx(&r.bar[s], kStageBytes);
  bulk_g2s(r.buf + s * kStageBytes, src, kStageBytes, &r.bar[s], policy);
}

// Stage the bf16 activations of SLOTS token slots over columns [col0, col0 +
// 64*nchunks) into shared memory as f16, each slot rescaled by 2^sigma[slot]
// (sigma from the slot's amax over the same columns, see pow2_rescale_exponent).
// tok_row(slot) gives the source row of x (or -1 for an empty slot); k = row length.
// Work items are (slot, 8-column group): one 16-byte load each, kStageBatch loads
// in flight per thread.  Pass 1 takes the per-slot amax (shared-memory atomicMax
// on the float bits, exact), pass 2 reloads (L1/L2 hits), converts and stores in
// the MMA fragment layout or the CUDA-core pair layout (see the constants above).
// All threads of the CTA call it; it ends with a __syncthreads.
constexpr int kStageBatch = 8;

template <bool kMMA, int SLOTS, typename TokRow>
__device__ __forceinline__ void stage_tokens(const uint16_t* __restrict__ x, int k, int col0, int nchunks,
                                             TokRow tok_row, unsigned* s_amax, int* sigma, uint8_t* xs) {
  const int groups = nchunks * 8;  // 8-column groups per slot
  const int items = SLOTS * groups;
  if (threadIdx.x < SLOTS) s_amax[threadIdx.x] = 0u;
  __syncthreads();
  auto src_of = [&](int it, int& slot, int& c8) -> const uint4* {
    slot = it / groups;
    c8 = it - slot * groups;
    const int col = col0 + c8 * 8;
    const int row = tok_row(slot);
    if (row < 0 || col >= k) return nullptr;
    return reinterpret_cast<const uint4*>(x + static_cast<size_t>(row) * k + col);
  };
  // ---- pass 1: amax per slot
  for (int base = threadIdx.x; base < items; base += blockDim.x * kStageBatch) {
    uint4 v[kStageBatch];
    int sl[kStageBatch];
#pragma unroll
    for (int j = 0; j < kStageBatch; ++j) {
      const int it = base + j * blockDim.x;
      int c8;
      const uint4* src = it < items ? src_of(it, sl[j], c8) : nullptr;
      v[j] = src ? __ldg(src) : make_uint4(0, 0, 0, 0);
      if (!src) sl[j] = -1;
    }
#pragma unroll
    for (int j = 0; j < kStageBatch; ++j) {
      if (sl[j] < 0) continue;
      const uint32_t w4[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
      float am = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        am = fmaxf(am, fmaxf(fabsf(__uint_as_float(w4[e] << 16)), fabsf(__uint_as_float(w4[e] & 0xFFFF0000u))));
      if (am > 0.f) atomicMax(&s_amax[sl[j]], __float_as_uint(am));
    }
  }
  __syncthreads();
  if (threadIdx.x < SLOTS) sigma[threadIdx.x] = pow2_rescale_exponent(__uint_as_float(s_amax[threadIdx.x]));
  __syncthreads();
  // ---- pass 2: convert and store
  uint32_t* xw = reinterpret_cast<uint32_t*>(xs);
  for (int base = threadIdx.x; base < items; base += blockDim.x * kStageBatch) {
    uint4 v[kStageBatch];
    int sl[kStageBatch], cg[kStageBatch];
#pragma unroll
    for (int j = 0; j < kStageBatch; ++j) {
      const int it = base + j * blockDim.x;
      sl[j] = -1;
      cg[j] = 0;
      v[j] = make_uint4(0, 0, 0, 0);
      if (it < items) {
        // empty slots and columns past k are stored as zeros (the tile padding
        // is zero too, but stale shared memory could hold non-finite values)
        const uint4* src = src_of(it, sl[j], cg[j]);
        if (src) v[j] = __ldg(src);
      }
    }
#pragma unroll
    for (int j = 0; j < kStageBatch; ++j) {
      if (sl[j] < 0) continue;  // past the last item
      const float sc = exp2i(sigma[sl[j]]);
      const uint32_t w4[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
      uint32_t h[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(w4[e] << 16) * sc, hi = __uint_as_float(w4[e] & 0xFFFF0000u) * sc;
        h[e] = static_cast<uint32_t>(f32_to_f16_bits(lo)) | (static_cast<uint32_t>(f32_to_f16_bits(hi)) << 16);
      }
      const int kcl = cg[j] >> 3, c64 = (cg[j] & 7) * 8;  // chunk, first column within the chunk
      if constexpr (kMMA) {
        constexpr int NT = (SLOTS + 7) / 8;
        // columns c64..c64+7 = k-tile kt, half hf, pairs t = 0..3 -> lanes (g, t), word 2*kt + hf
        const int kt = c64 >> 4, hf = (c64 >> 3) & 1;
        const int nt = sl[j] >> 3, g = sl[j] & 7;
        uint32_t* dst = xw + (static_cast<size_t>(kcl) * NT + nt) * 256 + (g * 4) * 8 + kt * 2 + hf;
#pragma unroll
        for (int t = 0; t < 4; ++t) dst[t * 8] = h[t];
      } else {
        uint4* dst = reinterpret_cast<uint4*>(xw + (static_cast<size_t>(kcl) * SLOTS + sl[j]) * 32 + c64 / 2);
        *dst = make_uint4(h[0], h[1], h[2], h[3]);
      }
    }
  }
  __syncthreads();
}

}  // namespace nvfp4
