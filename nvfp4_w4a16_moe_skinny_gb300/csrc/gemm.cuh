// Dense skinny NVFP4 GEMM (M <= 16) and the lm_head with fused argmax.
//
// y[m, n] = sum_k w_hat[n, k] x[m, k] -- gemma-cuda-hybrid README, "Everything
// it has / Inference engine" (one GEMM for every M<=16 product, including both
// lm_heads; greedy argmax is bit-exact: "Headline numbers").
//
// Work decomposition (one CTA of 16 warps per SM):
//  * K is cut into `csplit` slices across CTAs (csplit = 1 for the lm_head);
//    CTA b takes k-slice b % csplit and row-block group b / csplit.  The
//    row-blocks (16 rows) of a group are dealt to the CTA's warps round-robin;
//    a warp streams its row-block's tiles of the k-slice through its own ring.
//  * csplit > 1: each CTA writes fp32 partials; the last CTA of a group to
//    arrive (one atomic ticket per group, no spinning) sums the csplit
//    partials in slice order and writes bf16 y.
//  * lm_head: each lane keeps the best (value, row) per token; warps and CTAs
//    reduce in fixed order (ties -> lower row); the last CTA to arrive writes
//    the result.  No logit leaves the SM.
#pragma once

#include "stream.cuh"

namespace nvfp4 {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;

enum { kEpiStore = 0, kEpiArgmax = 1 };

struct SkinnyParams {
  const uint8_t* w;      // repacked matrix
  const float* gscale;   // &g
  const uint16_t* x;     // [m, k] bf16
  int m, n, k;
  int nb, kc;            // padded 16-row blocks, 64-column chunks
  int csplit, ngroups;   // grid = csplit * ngroups
  int ns;                // ring stages per warp
  uint16_t* y;           // [m, n] bf16 (store)
  float* partial;        // [csplit][m][nb*16] fp32 (csplit > 1)
  unsigned* counters;    // [ngroups] (store, csplit > 1) or [1] (argmax)
  float* am_val;         // [grid][m] (argmax)
  int* am_idx;           // [grid][m]
  float* max_logit;      // [m]
  int* argmax;           // [m]
};

__host__ __device__ inline int kslice_lo(int kc, int csplit, int s) {
  return static_cast<int>((static_cast<long long>(kc) * s) / csplit);
}

// Shared-memory bytes for one CTA (also used by the host).
__host__ __device__ inline size_t skinny_smem_bytes(bool mma, int slots, int kcs_max, int ns) {
  const int nt = (slots + 7) / 8;
  const size_t ring = static_cast<size_t>(kWarps) * ns * kStageBytes;
  const size_t bars = static_cast<size_t>(kWarps) * ns * 8;
  const size_t xs = mma ? static_cast<size_t>(nt) * kcs_max * kXFragChunkBytes
                        : static_cast<size_t>(slots) * kcs_max * kXCoreChunkBytes;
  const size_t misc = 16 * 4 + 16 * 4 + kWarps * 16 * 8 + 16;  // sigma, mul, argmax scratch, flag
  return ring + bars + xs + misc;
}

__device__ __forceinline__ bool better(float v, int r, float bv, int br) {
  return v > bv || (v == bv && r < br);
}

template <int MT, bool kMMA, int kEpi>
__global__ void __launch_bounds__(kThreads, 1) skinny_kernel(const SkinnyParams p) {
  constexpr int NT = (MT + 7) / 8;
  constexpr int SLOTS = kMMA ? NT * 8 : MT;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = blockIdx.x / p.csplit, ks = blockIdx.x - gi * p.csplit;
  const int kc0 = kslice_lo(p.kc, p.csplit, ks), kc1 = kslice_lo(p.kc, p.csplit, ks + 1);
  const int kcs = kc1 - kc0;
  const int kcs_max = (p.kc + p.csplit - 1) / p.csplit;
  const int rb0 = kslice_lo(p.nb, p.ngroups, gi), rb1 = kslice_lo(p.nb, p.ngroups, gi + 1);

  const size_t ring_bytes = static_cast<size_t>(kWarps) * p.ns * kStageBytes;
  Ring ring{smem + static_cast<size_t>(warp) * p.ns * kStageBytes,
            reinterpret_cast<uint64_t*>(smem + ring_bytes) + warp * p.ns, p.ns};
  uint8_t* xs = smem + ring_bytes + static_cast<size_t>(kWarps) * p.ns * 8;
  const size_t xs_bytes = kMMA ? static_cast<size_t>(NT) * kcs_max * kXFragChunkBytes
                               : static_cast<size_t>(SLOTS) * kcs_max * kXCoreChunkBytes;
  int* sigma = reinterpret_cast<int*>(xs + xs_bytes);
  float* mul = reinterpret_cast<float*>(sigma + 16);
  float* red_v = mul + 16;
  int* red_i = reinterpret_cast<int*>(red_v + kWarps * 16);
  int* flag = red_i + kWarps * 16;

  // this warp's units: row-blocks rb0 + warp + i * kWarps
  const int n_units = (rb1 - rb0 > warp) ? (rb1 - rb0 - warp + kWarps - 1) / kWarps : 0;
  const int cpu = (kcs + kTPS - 1) / kTPS;  // chunks per unit
  const int n_chunks = n_units * cpu;
  const uint64_t policy = l2_evict_first_policy();
  auto chunk_src = [&](int q, int& ntl) -> const uint8_t* {
    const int u = q / cpu, c = q - u * cpu;
    const int rb = rb0 + warp + u * kWarps;
    ntl = min(kTPS, kcs - c * kTPS);
    return p.w + (static_cast<size_t>(rb) * p.kc + kc0 + c * kTPS) * kTileBytes;
  };

  ring_init(ring, lane);
  if (lane == 0) {
    const int pre = min(p.ns, n_chunks);
    for (int q = 0; q < pre; ++q) {
      int ntl;
      const uint8_t* src = chunk_src(q, ntl);
      ring_issue(ring, q, src, ntl, policy);
    }
  }

  // activations of this CTA's k-slice -> shared memory (f16, per-token 2^sigma)
  const int col_lo = kc0 * kTileK, col_hi = min(kc1 * kTileK, p.k);
  auto tok_row = [&](int slot) -> int { return slot < p.m ? slot : -1; };
  (void)col_hi;
  stage_tokens<kMMA, SLOTS>(p.x, p.k, col_lo, kcs, tok_row, reinterpret_cast<unsigned*>(red_v), sigma, xs);
  if (threadIdx.x < SLOTS) mul[threadIdx.x] = __ldg(p.gscale) * exp2i(8 - sigma[threadIdx.x]);
  __syncthreads();

  const int g = lane >> 2, t4 = lane & 3;
  float accm[NT][4];
  float accc[MT][2];
  float bv[kMMA ? NT * 2 : MT];
  int bi[kMMA ? NT * 2 : MT];
#pragma unroll
  for (int i = 0; i < (kMMA ? NT * 2 : MT); ++i) bv[i] = -INFINITY, bi[i] = 0x7FFFFFFF;
  auto zero_acc = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) accm[nt][i] = 0.f;
#pragma unroll
    for (int m = 0; m < MT; ++m) accc[m][0] = accc[m][1] = 0.f;
  };
  zero_acc();

  int q_fail = -1;
  for (int q = 0; q < n_chunks; ++q) {
    const int s = q % p.ns;
    const uint32_t parity = static_cast<uint32_t>(q / p.ns) & 1u;
    if (!mbar_wait_warp(&ring.bar[s], parity)) {
      q_fail = q;
      break;
    }
    const int u = q / cpu, c = q - u * cpu;
    const int t0 = c * kTPS;
    const int ntl = min(kTPS, kcs - t0);
    const uint8_t* st = ring.buf + s * kStageBytes;
#pragma unroll
    for (int j = 0; j < kTPS; ++j) {
      if (j < ntl) {
        if constexpr (kMMA) {
          mma_tile<NT>(st + j * kTileBytes, xs + static_cast<size_t>(t0 + j) * NT * kXFragChunkBytes, lane, accm);
        } else {
          core_tile<MT>(st + j * kTileBytes, xs + static_cast<size_t>(t0 + j) * MT * kXCoreChunkBytes, g, t4, accc);
        }
      }
    }
    __syncwarp();
    if (lane == 0 && q + p.ns < n_chunks) {
      fence_proxy_async_smem();
      int ntl2;
      const uint8_t* src = chunk_src(q + p.ns, ntl2);
      ring_issue(ring, s, src, ntl2, policy);
    }
    if (c == cpu - 1) {
      // ---- end of a row-block: epilogue
      const int rb = rb0 + warp + u * kWarps;
      if constexpr (!kMMA) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            float v = accc[m][r];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            accc[m][r] = v;
          }
      }
      if constexpr (kEpi == kEpiStore) {
        if constexpr (kMMA) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int row = rb * 16 + g + 8 * (i >> 1);
              const int tok = nt * 8 + 2 * t4 + (i & 1);
              if (tok < p.m && row < p.n) {
                const float v = accm[nt][i] * mul[tok];
                if (p.csplit == 1)
                  p.y[static_cast<size_t>(tok) * p.n + row] = f32_to_bf16_bits(v);
                else
                  p.partial[(static_cast<size_t>(ks) * p.m + tok) * (p.nb * 16) + row] = v;
              }
            }
        } else {
          if (t4 == 0) {
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                const int row = rb * 16 + g + 8 * r;
                if (m < p.m && row < p.n) {
                  const float v = accc[m][r] * mul[m];
                  if (p.csplit == 1)
                    p.y[static_cast<size_t>(m) * p.n + row] = f32_to_bf16_bits(v);
                  else
                    p.partial[(static_cast<size_t>(ks) * p.m + m) * (p.nb * 16) + row] = v;
                }
              }
          }
        }
      } else {  // argmax: raw accumulators compare like logits (positive per-token multiplier)
        if constexpr (kMMA) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int row = rb * 16 + g + 8 * (i >> 1);
              const int slot = nt * 2 + (i & 1);
              if (row < p.n && better(accm[nt][i], row, bv[slot], bi[slot])) bv[slot] = accm[nt][i], bi[slot] = row;
            }
        } else {
#pragma unroll
          for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int row = rb * 16 + g + 8 * r;
              if (row < p.n && better(accc[m][r], row, bv[m], bi[m])) bv[m] = accc[m][r], bi[m] = row;
            }
        }
      }
      zero_acc();
    }
  }
  if (q_fail >= 0) {
    // a copy did not complete in time: wait (bounded) for the copies this warp
    // still has in flight so none lands after the CTA exits, then give up
    const int q_end = min(q_fail + p.ns, n_chunks);
    for (int q = q_fail + 1; q < q_end; ++q) (void)mbar_wait_warp(&ring.bar[q % p.ns], static_cast<uint32_t>(q / p.ns) & 1u);
    __syncwarp();
  }

  if constexpr (kEpi == kEpiStore) {
    if (p.csplit > 1) {
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) {
        const unsigned ticket = atomicAdd(&p.counters[gi], 1u);
        const int last = ticket == static_cast<unsigned>(p.csplit - 1);
        if (last) atomicExch(&p.counters[gi], 0u);
        *flag = last;
      }
      __syncthreads();
      if (*flag) {
        __threadfence();
        const int r0 = rb0 * 16, r1 = min(rb1 * 16, p.n);
        const int rows = r1 - r0;
        const size_t stride = static_cast<size_t>(p.m) * p.nb * 16;
        for (int i = threadIdx.x; i < rows * p.m; i += blockDim.x) {
          const int tok = i / rows, row = r0 + (i - tok * rows);
          const float* src = p.partial + static_cast<size_t>(tok) * p.nb * 16 + row;
          float acc = 0.f;
          for (int s = 0; s < p.csplit; ++s) acc += __ldcg(src + s * stride);
          p.y[static_cast<size_t>(tok) * p.n + row] = f32_to_bf16_bits(acc);
        }
      }
    }
  } else {
    // ---- argmax: lanes -> warp
    if constexpr (kMMA) {
#pragma unroll
      for (int slot = 0; slot < NT * 2; ++slot) {
        float v = bv[slot];
        int r = bi[slot];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, v, off);
          const int orow = __shfl_xor_sync(0xffffffffu, r, off);
          if (better(ov, orow, v, r)) v = ov, r = orow;
        }
        if (g == 0) {
          const int tok = (slot >> 1) * 8 + 2 * t4 + (slot & 1);
          red_v[warp * 16 + tok] = v;
          red_i[warp * 16 + tok] = r;
        }
      }
    } else {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float v = bv[m];
        int r = bi[m];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, v, off);
          const int orow = __shfl_xor_sync(0xffffffffu, r, off);
          if (better(ov, orow, v, r)) v = ov, r = orow;
        }
        if (lane == 0) red_v[warp * 16 + m] = v, red_i[warp * 16 + m] = r;
      }
    }
    __syncthreads();
    // ---- warps -> CTA (fixed order), scaled to logits
    if (threadIdx.x < p.m) {
      const int tok = threadIdx.x;
      float v = -INFINITY;
      int r = 0x7FFFFFFF;
      for (int w = 0; w < kWarps; ++w)
        if (better(red_v[w * 16 + tok], red_i[w * 16 + tok], v, r)) v = red_v[w * 16 + tok], r = red_i[w * 16 + tok];
      p.am_val[static_cast<size_t>(blockIdx.x) * p.m + tok] = (r == 0x7FFFFFFF) ? -INFINITY : v * mul[tok];
      p.am_idx[static_cast<size_t>(blockIdx.x) * p.m + tok] = r;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned ticket = atomicAdd(&p.counters[0], 1u);
      const int last = ticket == gridDim.x - 1;
      if (last) atomicExch(&p.counters[0], 0u);
      *flag = last;
    }
    __syncthreads();
    if (*flag && threadIdx.x < p.m) {
      __threadfence();
      const int tok = threadIdx.x;
      float v = -INFINITY;
      int r = 0x7FFFFFFF;
      for (unsigned b = 0; b < gridDim.x; ++b) {
        const float ov = __ldcg(p.am_val + static_cast<size_t>(b) * p.m + tok);
        const int orow = __ldcg(p.am_idx + static_cast<size_t>(b) * p.m + tok);
        if (better(ov, orow, v, r)) v = ov, r = orow;
      }
      p.max_logit[tok] = v;
      p.argmax[tok] = r;
    }
  }
}

}  // namespace nvfp4
