// Grouped MoE FFN with NVFP4 experts: router top-k, expert grouping, grouped
// gate+up with the GELU-tanh gate fused in the epilogue, grouped down, and a
// fixed-order combine.
//
// TensorSharp docs/models/gemma4.md: "3.2 Per-layer (MoE)" and "4.6 MoE" (router
// logits -> softmax -> top-k; each chosen expert runs its gated FFN; weighted
// sum), "3.1 Per-layer (dense)" ([gate || up] from the fused matmul, GELU on the
// gate, times up, then down), "14. Optimization opportunities / Completed
// (Expert-batched FFN)" (the whole layer as grouped gate+up / down products over
// stacked 3-D expert weights with a fused GEGLU and an aggregation).
// gemma-cuda-hybrid README, "Everything it has / Inference engine": grouped
// weight-resident MoE with no atomics.  TensorFold issue #1048, "Steps", step 2:
// GELU-tanh.
#pragma once

#include "gemm.cuh"

namespace nvfp4 {

// ------------------------------------------------------------------ router

// One CTA.  Phase 1: one warp per token selects the top_k largest logits
// (descending, ties -> lower expert id) by repeated warp arg-max and takes a
// softmax over them.  Phase 2: a stable counting sort of the (token, slot)
// pairs by expert with warp ballots: counts, an exclusive scan, then ranked
// writes in ascending pair order.  No atomics.
constexpr int kRouteThreads = 1024;

__global__ void __launch_bounds__(kRouteThreads, 1)
    moe_route_kernel(const float* __restrict__ logits, int m, int n_experts, int top_k, int* __restrict__ ids,
                     float* __restrict__ probs, int* __restrict__ offsets, int* __restrict__ sorted_pairs) {
  extern __shared__ int route_smem[];
  int* s_ids = route_smem;                 // [m * top_k]
  int* s_cnt = s_ids + m * top_k;          // [n_experts + 1]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int pairs = m * top_k;
  for (int t = warp; t < m; t += nwarps) {
    const float* row = logits + static_cast<size_t>(t) * n_experts;
    uint32_t taken = 0;  // bit i: expert lane + 32*i already chosen (n_experts <= 1024)
    float chosen_v[32];
    int chosen_e[32];
    for (int r = 0; r < top_k; ++r) {
      float bv = -INFINITY;
      int be = 0x7FFFFFFF;
      for (int i = 0; i * 32 < n_experts; ++i) {
        const int e = lane + 32 * i;
        if (e < n_experts && !((taken >> i) & 1u)) {
          const float v = __ldg(row + e);
          if (v > bv || (v == bv && e < be)) bv = v, be = e;
        }
      }
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oe = __shfl_xor_sync(0xffffffffu, be, off);
        if (ov > bv || (ov == bv && oe < be)) bv = ov, be = oe;
      }
      if (lane == (be & 31)) taken |= 1u << (be >> 5);
      chosen_v[r] = bv;
      chosen_e[r] = be;
    }
    // softmax over the chosen logits (chosen_v[0] is the maximum)
    if (lane < top_k) {
      float z = 0.f;
      float mine = 0.f;
      for (int r = 0; r < top_k; ++r) {
        const float ez = expf(chosen_v[r] - chosen_v[0]);
        z += ez;
        if (r == lane) mine = ez;
      }
      ids[t * top_k + lane] = chosen_e[lane];
      probs[t * top_k + lane] = mine / z;
      s_ids[t * top_k + lane] = chosen_e[lane];
    }
  }
  __syncthreads();
  // counts per expert (warp per expert, ballots over the pairs)
  for (int e = warp; e < n_experts; e += nwarps) {
    int cnt = 0;
    for (int base = 0; base < pairs; base += 32) {
      const int pidx = base + lane;
      const bool hit = pidx < pairs && s_ids[pidx] == e;
      cnt += __popc(__ballot_sync(0xffffffffu, hit));
    }
    if (lane == 0) s_cnt[e] = cnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int e = 0; e < n_experts; ++e) {
      const int c = s_cnt[e];
      s_cnt[e] = run;
      offsets[e] = run;
      run += c;
    }
    s_cnt[n_experts] = run;
    offsets[n_experts] = run;
  }
  __syncthreads();
  // ranked writes in ascending pair order
  for (int e = warp; e < n_experts; e += nwarps) {
    int pos = s_cnt[e];
    for (int base = 0; base < pairs; base += 32) {
      const int pidx = base + lane;
      const bool hit = pidx < pairs && s_ids[pidx] == e;
      const uint32_t mask = __ballot_sync(0xffffffffu, hit);
      if (hit) sorted_pairs[pos + __popc(mask & ((1u << lane) - 1u))] = pidx;
      pos += __popc(mask);
    }
  }
}

// ------------------------------------------------------------------ grouped FFN

enum { kEpiGatedGelu = 0, kEpiPartial = 1 };
constexpr int kSharedSeg = -1;  // segment id of the always-on shared expert

struct MoEParams {
  const uint8_t* w;        // stacked routed matrices [E]
  const float* gs;         // [E]
  const uint8_t* w_sh;     // shared matrix or nullptr
  const float* gs_sh;
  size_t mat_bytes;        // repacked bytes of one matrix
  const uint16_t* x;       // activations: x [m, d] (gate_up) or h [pairs_total, inter] (down)
  int k;                   // columns of one matrix = activation row length
  int nb, kc;              // row-blocks, 64-column chunks of one matrix
  int m, top_k, n_experts;
  const int* offsets;      // [E + 1]
  const int* pairs;        // [m * top_k]
  uint16_t* h_out;         // gate_up epilogue: h [pairs_total, inter]
  float* d_out;            // down epilogue: [pairs_total, d_out_cols]
  int out_cols;            // inter (gate_up) or d (down)
  int ns;
};

__device__ __forceinline__ float gelu_tanh(float z) {
  // 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))
  const float u = 0.7978845608028654f * fmaf(0.044715f * z, z * z, z);
  return 0.5f * z * (1.0f + tanhf(u));
}

__host__ __device__ inline size_t moe_smem_bytes(bool mma, int slots, int kc, int ns, int n_experts) {
  const int nt = (slots + 7) / 8;
  const size_t ring = static_cast<size_t>(kWarps) * ns * kStageBytes;
  const size_t bars = static_cast<size_t>(kWarps) * ns * 8;
  const size_t xs = mma ? static_cast<size_t>(nt) * kc * kXFragChunkBytes : static_cast<size_t>(slots) * kc * kXCoreChunkBytes;
  const size_t misc = 16 * 4 * 5 + (static_cast<size_t>(n_experts) + 2) * 4 + 16;
  return ring + bars + xs + misc;
}

// One CTA of 16 warps per SM.  The work items are (segment, row-block) where the
// segments are the experts that received tokens (ascending id) followed by the
// shared expert; every segment has the same nb row-blocks, so item i is
// (i / nb, i % nb).  CTA b takes a contiguous, balanced range of items.  Within
// a segment the CTA's row-blocks are dealt to its warps round-robin; at a
// segment boundary the CTA stages the next segment's tokens (one barrier),
// while every warp's ring keeps prefetching weights across the boundary.
template <int MT, bool kMMA, int kEpi>
__global__ void __launch_bounds__(kThreads, 1) moe_ffn_kernel(const MoEParams p) {
  constexpr int NT = (MT + 7) / 8;
  constexpr int SLOTS = kMMA ? NT * 8 : MT;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const size_t ring_bytes = static_cast<size_t>(kWarps) * p.ns * kStageBytes;
  Ring ring{smem + static_cast<size_t>(warp) * p.ns * kStageBytes,
            reinterpret_cast<uint64_t*>(smem + ring_bytes) + warp * p.ns, p.ns};
  uint8_t* xs = smem + ring_bytes + static_cast<size_t>(kWarps) * p.ns * 8;
  const size_t xs_bytes = kMMA ? static_cast<size_t>(NT) * p.kc * kXFragChunkBytes
                               : static_cast<size_t>(SLOTS) * p.kc * kXCoreChunkBytes;
  int* sigma = reinterpret_cast<int*>(xs + xs_bytes);
  float* mul = reinterpret_cast<float*>(sigma + 16);
  int* slot_row = reinterpret_cast<int*>(mul + 16);   // activation row of each token slot
  int* slot_out = slot_row + 16;                      // output row (pair index) of each slot
  unsigned* s_amax = reinterpret_cast<unsigned*>(slot_out + 16);
  int* seg_list = reinterpret_cast<int*>(s_amax + 16);  // [n_experts + 1]
  int* n_seg_s = seg_list + p.n_experts + 1;

  // ---- active segments (warp 0, ballots in ascending expert order)
  if (warp == 0) {
    int n = 0;
    for (int base = 0; base < p.n_experts; base += 32) {
      const int e = base + lane;
      const bool act = e < p.n_experts && __ldg(p.offsets + e + 1) > __ldg(p.offsets + e);
      const uint32_t mask = __ballot_sync(0xffffffffu, act);
      if (act) seg_list[n + __popc(mask & ((1u << lane) - 1u))] = e;
      n += __popc(mask);
    }
    if (lane == 0) {
      if (p.w_sh) seg_list[n++] = kSharedSeg;
      *n_seg_s = n;
    }
  }
  __syncthreads();
  const int n_seg = *n_seg_s;
  const long long n_items = static_cast<long long>(n_seg) * p.nb;
  const int it0 = static_cast<int>(n_items * blockIdx.x / gridDim.x);
  const int it1 = static_cast<int>(n_items * (blockIdx.x + 1) / gridDim.x);
  if (it0 >= it1) return;
  const int seg0 = it0 / p.nb, seg1 = (it1 - 1) / p.nb;  // inclusive
  const int cpu = (p.kc + kTPS - 1) / kTPS;

  // run r = segment seg0 + r, items [max(it0, s*nb), min(it1, (s+1)*nb))
  auto run_lo = [&](int r) { return max(it0, (seg0 + r) * p.nb); };
  auto run_hi = [&](int r) { return min(it1, (seg0 + r + 1) * p.nb); };
  auto run_units = [&](int r) {
    const int len = run_hi(r) - run_lo(r);
    return len > warp ? (len - warp + kWarps - 1) / kWarps : 0;
  };
  auto matrix_of = [&](int seg) -> const uint8_t* {
    const int e = seg_list[seg];
    return e == kSharedSeg ? p.w_sh : p.w + static_cast<size_t>(e) * p.mat_bytes;
  };
  const int n_runs = seg1 - seg0 + 1;
  // producer cursor (lane 0): run, unit, chunk
  int pr = 0, pu = 0, pc = 0;
  auto prod_skip = [&]() {
    while (pr < n_runs && pu >= run_units(pr)) pu = 0, ++pr;
  };
  const uint64_t policy = l2_evict_first_policy();
  auto prod_issue = [&](int stage) {
    const int item = run_lo(pr) + warp + pu * kWarps;
    const int rb = item - (seg0 + pr) * p.nb;
    const int ntl = min(kTPS, p.kc - pc * kTPS);
    const uint8_t* src = matrix_of(seg0 + pr) + (static_cast<size_t>(rb) * p.kc + pc * kTPS) * kTileBytes;
    ring_issue(ring, stage, src, ntl, policy);
    if (++pc == cpu) pc = 0, ++pu, prod_skip();
  };
  ring_init(ring, lane);
  int total_chunks = 0;
  for (int r = 0; r < n_runs; ++r) total_chunks += run_units(r) * cpu;
  if (lane == 0) {
    prod_skip();
    for (int q = 0; q < min(p.ns, total_chunks); ++q) prod_issue(q);
  }

  const int g = lane >> 2, t4 = lane & 3;
  float accm[NT][4];
  float accc[MT][2];
  int q = 0;
  int q_fail = -1;
  // every warp runs every iteration of this loop (its barriers are CTA-wide); a
  // warp whose copy timed out only skips its own tiles
  for (int r = 0; r < n_runs; ++r) {
    const int seg = seg0 + r;
    const int e = seg_list[seg];
    // ---- stage this segment's tokens
    __syncthreads();
    if (threadIdx.x < 16) {
      const int j = threadIdx.x;
      int row = -1, out = -1;
      if (e == kSharedSeg) {
        if (j < p.m) out = p.m * p.top_k + j, row = (kEpi == kEpiGatedGelu) ? j : out;
      } else {
        const int lo = __ldg(p.offsets + e), cnt = __ldg(p.offsets + e + 1) - lo;
        if (j < cnt) {
          out = __ldg(p.pairs + lo + j);
          row = (kEpi == kEpiGatedGelu) ? out / p.top_k : out;
        }
      }
      slot_row[j] = j < SLOTS ? row : -1;
      slot_out[j] = j < SLOTS ? out : -1;
    }
    __syncthreads();
    auto tok_row = [&](int slot) -> int { return slot_row[slot]; };
    stage_tokens<kMMA, SLOTS>(p.x, p.k, 0, p.kc, tok_row, s_amax, sigma, xs);
    if (threadIdx.x < SLOTS) {
      const float gsc = (e == kSharedSeg) ? __ldg(p.gs_sh) : __ldg(p.gs + e);
      mul[threadIdx.x] = gsc * exp2i(8 - sigma[threadIdx.x]);
    }
    __syncthreads();

    const int lo = run_lo(r);
    const int units = run_units(r);
    for (int u = 0; u < units && q_fail < 0; ++u) {
      const int rb = lo + warp + u * kWarps - seg * p.nb;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) accm[nt][i] = 0.f;
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) accc[mm][0] = accc[mm][1] = 0.f;
      for (int c = 0; c < cpu; ++c, ++q) {
        const int s = q % p.ns;
        if (!mbar_wait_warp(&ring.bar[s], static_cast<uint32_t>(q / p.ns) & 1u)) {
          q_fail = q;
          break;
        }
        const int t0 = c * kTPS;
        const int ntl = min(kTPS, p.kc - t0);
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
        if (lane == 0 && q + p.ns < total_chunks) {
          fence_proxy_async_smem();
          prod_issue(s);
        }
      }
      if (q_fail >= 0) break;
      // ---- epilogue of row-block rb of this segment
      if constexpr (!kMMA) {
#pragma unroll
        for (int mm = 0; mm < MT; ++mm)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            float v = accc[mm][rr];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            accc[mm][rr] = v;
          }
      }
      if constexpr (kEpi == kEpiGatedGelu) {
        // gated layout: rows g = gate i, g+8 = up i, with i = rb*8 + g
        const int i = rb * 8 + g;
        if constexpr (kMMA) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int slot = nt * 8 + 2 * t4 + hf;
              const int out = slot_out[slot];
              if (out >= 0) {
                const float gate = accm[nt][hf] * mul[slot], up = accm[nt][2 + hf] * mul[slot];
                p.h_out[static_cast<size_t>(out) * p.out_cols + i] = f32_to_bf16_bits(gelu_tanh(gate) * up);
              }
            }
        } else {
          if (t4 == 0) {
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
              const int out = slot_out[mm];
              if (out >= 0) {
                const float gate = accc[mm][0] * mul[mm], up = accc[mm][1] * mul[mm];
                p.h_out[static_cast<size_t>(out) * p.out_cols + i] = f32_to_bf16_bits(gelu_tanh(gate) * up);
              }
            }
          }
        }
      } else {
        if constexpr (kMMA) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int slot = nt * 8 + 2 * t4 + (i & 1);
              const int row = rb * 16 + g + 8 * (i >> 1);
              const int out = slot_out[slot];
              if (out >= 0 && row < p.out_cols)
                p.d_out[static_cast<size_t>(out) * p.out_cols + row] = accm[nt][i] * mul[slot];
            }
        } else {
          if (t4 == 0) {
#pragma unroll
            for (int mm = 0; mm < MT; ++mm)
#pragma unroll
              for (int rr = 0; rr < 2; ++rr) {
                const int row = rb * 16 + g + 8 * rr;
                const int out = slot_out[mm];
                if (out >= 0 && row < p.out_cols)
                  p.d_out[static_cast<size_t>(out) * p.out_cols + row] = accc[mm][rr] * mul[mm];
              }
          }
        }
      }
    }
  }
  if (q_fail >= 0) {
    const int q_end = min(q_fail + p.ns, total_chunks);
    for (int qq = q_fail + 1; qq < q_end; ++qq)
      (void)mbar_wait_warp(&ring.bar[qq % p.ns], static_cast<uint32_t>(qq / p.ns) & 1u);
  }
}

// out[t, j] = bf16( sum_r probs[t, r] * d[t*top_k + r, j] + d[m*top_k + t, j] ), fixed order.
__global__ void moe_combine_kernel(const float* __restrict__ d, const float* __restrict__ probs, int m, int top_k,
                                   int cols, bool shared, uint16_t* __restrict__ out) {
  const size_t total = static_cast<size_t>(m) * cols;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / cols), j = static_cast<int>(i - static_cast<size_t>(t) * cols);
    float acc = 0.f;
    for (int r = 0; r < top_k; ++r)
      acc = fmaf(__ldg(probs + t * top_k + r), __ldg(d + static_cast<size_t>(t * top_k + r) * cols + j), acc);
    if (shared) acc += __ldg(d + static_cast<size_t>(m * top_k + t) * cols + j);
    out[i] = f32_to_bf16_bits(acc);
  }
}

}  // namespace nvfp4
