// MoE router (top-k, softmax, expert grouping) and the fixed-order combine of the
// grouped expert FFN; the grouped gate+up (GELU-tanh fused in the epilogue) and
// down products run on the streaming kernel of kernel.cuh.
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

#include "kernel.cuh"

namespace nvfp4 {

// ------------------------------------------------------------------ router

// Phase 1: one warp per token selects the top_k largest logits (descending,
// ties -> lower expert id) by repeated warp arg-max and takes a softmax over
// them; lane r keeps the r-th choice.  Phase 2: a stable counting sort of the
// (token, slot) pairs by expert: counts, a block-wide exclusive scan, then
// ranked writes in ascending pair order.  No atomics.  A decode batch (m <= 32)
// runs both phases in one CTA; a larger batch runs phase 1 over many CTAs and
// phase 2 in one.  NPER: logits per lane (n_experts <= 32 * NPER).
constexpr int kRouteThreads = 1024;

// Routing weight options (moe_route_topk_ex): the softmax over all experts read
// at the chosen ones (not renormalised over the top_k).
constexpr int kRouteSoftmaxAll = 1;

// Top-k + softmax of token t by one warp; lane r < top_k writes the r-th choice
// (and, when s_ids is given, also into shared memory).  With kRouteSoftmaxAll the
// denominator sums every expert's exp; escale (nullable) scales each weight by
// its expert's entry.
template <int NPER>
__device__ __forceinline__ void token_topk(const float* __restrict__ logits, int t, int n_experts, int top_k, int lane,
                                           int* __restrict__ ids, float* __restrict__ probs, int* s_ids, int flags,
                                           const float* __restrict__ escale) {
  {
    const float* row = logits + static_cast<size_t>(t) * n_experts;
    // experts lane + 32*i, read once, as 64-bit keys (pack_value_row: larger logit,
    // then lower id, is larger); a NaN logit counts as -inf; 0 (below every valid
    // key) marks an expert that does not exist or was already chosen
    float lv[NPER];
    unsigned long long key[NPER];
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
      const int e = lane + 32 * i;
      const float v = e < n_experts ? __ldg(row + e) : -INFINITY;
      lv[i] = v == v ? v : -INFINITY;
      key[i] = e < n_experts ? pack_value_row(lv[i], e) : 0ull;
    }
    // top_k rounds of a warp-wide maximum: each round's winner is a valid expert not
    // chosen before (top_k <= n_experts): when all that remain are -inf, the lowest id
    float myv = -INFINITY;
    int mye = 0;
    for (int r = 0; r < top_k; ++r) {
      unsigned long long best = 0ull;
#pragma unroll
      for (int i = 0; i < NPER; ++i) best = key[i] > best ? key[i] : best;
      unsigned long long wmax = best;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, wmax, off);
        wmax = o > wmax ? o : wmax;
      }
#pragma unroll
      for (int i = 0; i < NPER; ++i)
        if (key[i] == wmax) key[i] = 0ull;  // keys are distinct: only the winner matches
      if (lane == r) myv = unpack_value(wmax), mye = unpack_row(wmax);
    }
    // softmax over the chosen logits, or over all of them (round 0 holds the maximum);
    // a token whose logits are all -inf (or NaN) gets weight 0 on every slot
    const float vmax = __shfl_sync(0xffffffffu, myv, 0);
    const bool none = vmax == -INFINITY;
    const float ez = lane < top_k && !none ? expf(myv - vmax) : 0.f;
    float z = ez;
    if (flags & kRouteSoftmaxAll) {
      z = 0.f;
#pragma unroll
      for (int i = 0; i < NPER; ++i)
        if (lane + 32 * i < n_experts && !none) z += expf(lv[i] - vmax);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    if (lane < top_k) {
      float pr = none ? 0.f : ez / z;
      if (escale) pr *= __ldg(escale + mye);
      ids[t * top_k + lane] = mye;
      probs[t * top_k + lane] = pr;
      if (s_ids) s_ids[t * top_k + lane] = mye;
    }
  }
}

// The stable counting sort of the pairs by expert by one warp (a decode batch:
// few pairs): per-expert counts from batches of 32 pairs (lanes holding the same
// expert find each other with a match; the group's first lane adds), an
// exclusive scan of the counts (each lane a contiguous run of experts), then the
// placement in the same batch order -- ascending pair order within an expert.
// No atomics, no block-wide barrier.  s_cnt: scratch of n_experts ints.
__device__ __forceinline__ void group_pairs_warp(const int* s_ids, int pairs, int n_experts, int* s_cnt, int lane,
                                                 int* __restrict__ offsets, int* __restrict__ sorted_pairs) {
  for (int e = lane; e < n_experts; e += 32) s_cnt[e] = 0;
  __syncwarp();
  for (int base = 0; base < pairs; base += 32) {
    const int q = base + lane;
    const int e = q < pairs ? s_ids[q] : -1 - lane;  // a lane past the end matches nobody
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    if (q < pairs && lane == __ffs(same) - 1) s_cnt[e] += __popc(same);
    __syncwarp();
  }
  // exclusive scan: lane l owns experts [l*per, (l+1)*per)
  const int per = (n_experts + 31) / 32;
  const int e0 = min(n_experts, lane * per), e1 = min(n_experts, e0 + per);
  int tot = 0;
  for (int e = e0; e < e1; ++e) tot += s_cnt[e];
  int incl = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  int run = incl - tot;
  for (int e = e0; e < e1; ++e) {
    const int c = s_cnt[e];
    offsets[e] = run;
    s_cnt[e] = run;  // now the next position of expert e
    run += c;
  }
  if (lane == 31) offsets[n_experts] = pairs;
  __syncwarp();
  for (int base = 0; base < pairs; base += 32) {
    const int q = base + lane;
    const int e = q < pairs ? s_ids[q] : -1 - lane;
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    if (q < pairs) sorted_pairs[s_cnt[e] + __popc(same & ((1u << lane) - 1u))] = q;
    __syncwarp();
    if (q < pairs && lane == __ffs(same) - 1) s_cnt[e] += __popc(same);
    __syncwarp();
  }
}

// The stable counting sort of the pairs by expert, from s_ids[pairs] in shared
// memory, by the whole CTA; s_cnt[n_experts + 1] and s_wsum[32] are scratch.
__device__ __forceinline__ void group_pairs(const int* s_ids, int pairs, int n_experts, int* s_cnt, int* s_wsum,
                                            int* __restrict__ offsets, int* __restrict__ sorted_pairs) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
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
  // exclusive scan of the counts: one thread per expert (n_experts <= 1024)
  const int c = threadIdx.x < n_experts ? s_cnt[threadIdx.x] : 0;
  int incl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? s_wsum[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += o;
    }
    s_wsum[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const int excl = incl - c + (warp > 0 ? s_wsum[warp - 1] : 0);
  if (threadIdx.x < n_experts) {
    s_cnt[threadIdx.x] = excl;
    offsets[threadIdx.x] = excl;
  }
  if (threadIdx.x == 0) offsets[n_experts] = pairs;
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

// The same sort for n_experts <= kHistExperts, in three passes over per-warp
// histograms (hist[w * n_experts + e], scratch of 32 * n_experts ints): warp w
// owns the contiguous pairs [w*C, (w+1)*C); (1) it counts its pairs per expert,
// lanes holding the same expert finding each other with a match; (2) thread e
// turns the counts into the first position of (expert e, warp w) -- expert-major,
// then warp, which is ascending pair order within an expert; (3) each warp walks
// its pairs again and places them.  No atomics; every count and position has a
// single writer.
constexpr int kHistExperts = 256;
// Shared-memory ints of the grouping's count scratch.
__host__ __device__ inline int route_scratch(int n_experts) {
  return n_experts <= kHistExperts ? 32 * n_experts : n_experts + 1;
}
__device__ __forceinline__ void group_pairs_hist(const int* s_ids, int pairs, int n_experts, int* hist, int* s_wsum,
                                                 int* __restrict__ offsets, int* __restrict__ sorted_pairs) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;  // 32
  const int per = (pairs + nwarps - 1) / nwarps;
  const int q0 = min(pairs, warp * per), q1 = min(pairs, q0 + per);
  for (int i = threadIdx.x; i < nwarps * n_experts; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  int* h = hist + warp * n_experts;
  for (int base = q0; base < q1; base += 32) {
    const int q = base + lane;
    const int e = q < q1 ? s_ids[q] : -1 - lane;  // a lane past the end matches nobody
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    if (q < q1 && lane == __ffs(same) - 1) h[e] += __popc(same);
    __syncwarp();
  }
  __syncthreads();
  // totals per expert, their exclusive scan (threads = experts), then the first
  // position of each (expert, warp)
  const int t = threadIdx.x;
  int total = 0;
  if (t < n_experts)
    for (int w = 0; w < nwarps; ++w) total += hist[w * n_experts + t];
  int incl = total;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  int excl = incl - total;
  for (int w = 0; w < warp; ++w) excl += s_wsum[w];
  if (t < n_experts) {
    offsets[t] = excl;
    int run = excl;
    for (int w = 0; w < nwarps; ++w) {
      const int c = hist[w * n_experts + t];
      hist[w * n_experts + t] = run;
      run += c;
    }
  }
  if (t == 0) offsets[n_experts] = pairs;
  __syncthreads();
  for (int base = q0; base < q1; base += 32) {
    const int q = base + lane;
    const int e = q < q1 ? s_ids[q] : -1 - lane;
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    if (q < q1) sorted_pairs[h[e] + __popc(same & ((1u << lane) - 1u))] = q;
    __syncwarp();
    if (q < q1 && lane == __ffs(same) - 1) h[e] += __popc(same);
    __syncwarp();
  }
}

// A decode batch: one CTA does both (one warp per token, then the grouping).
template <int NPER>
__global__ void __launch_bounds__(kRouteThreads, 1)
    moe_route_kernel(const float* __restrict__ logits, int m, int n_experts, int top_k, int flags,
                     const float* __restrict__ escale, int* __restrict__ ids, float* __restrict__ probs,
                     int* __restrict__ offsets, int* __restrict__ sorted_pairs) {
  extern __shared__ int route_smem[];
  const int pairs = m * top_k;
  int* s_ids = route_smem;                                  // [pairs]
  int* s_cnt = s_ids + pairs;                               // [route_scratch(n_experts)]
  int* s_wsum = s_cnt + route_scratch(n_experts);           // [32] per-warp totals of the scan
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  pdl_wait();  // the logits may come from the previous grid
  pdl_launch_dependents();
  for (int t = warp; t < m; t += nwarps)
    token_topk<NPER>(logits, t, n_experts, top_k, lane, ids, probs, s_ids, flags, escale);
  __syncthreads();
  // at most 32 tokens: one warp groups the pairs
  if (warp == 0) group_pairs_warp(s_ids, pairs, n_experts, s_cnt, lane, offsets, sorted_pairs);
  (void)s_wsum;
}

// A prefill chunk, step 1: the top-k of every token, one warp per token over
// many CTAs.
constexpr int kTopkWarps = 8;
template <int NPER>
__global__ void __launch_bounds__(kTopkWarps * 32)
    moe_topk_kernel(const float* __restrict__ logits, int m, int n_experts, int top_k, int flags,
                    const float* __restrict__ escale, int* __restrict__ ids, float* __restrict__ probs) {
  const int t = blockIdx.x * kTopkWarps + (threadIdx.x >> 5);
  pdl_wait();  // the logits may come from the previous grid
  pdl_launch_dependents();
  if (t < m) token_topk<NPER>(logits, t, n_experts, top_k, threadIdx.x & 31, ids, probs, nullptr, flags, escale);
}

// A prefill chunk, step 2: the grouping of all pairs by one CTA (the histogram
// sort when the experts allow it: the ballot sort scans every pair once per
// expert, ~4x slower at 4,096 pairs).
__global__ void __launch_bounds__(kRouteThreads, 1)
    moe_group_kernel(const int* __restrict__ ids, int pairs, int n_experts, int* __restrict__ offsets,
                     int* __restrict__ sorted_pairs) {
  extern __shared__ int route_smem[];
  int* s_ids = route_smem;                         // [pairs]
  int* s_cnt = s_ids + pairs;                      // [route_scratch(n_experts)]
  int* s_wsum = s_cnt + route_scratch(n_experts);  // [32]
  pdl_wait();  // the ids come from the previous grid
  pdl_launch_dependents();
  for (int q = threadIdx.x; q < pairs; q += blockDim.x) s_ids[q] = __ldg(ids + q);
  __syncthreads();
  if (n_experts <= kHistExperts)
    group_pairs_hist(s_ids, pairs, n_experts, s_cnt, s_wsum, offsets, sorted_pairs);
  else
    group_pairs(s_ids, pairs, n_experts, s_cnt, s_wsum, offsets, sorted_pairs);
}

// Router normalisation (TensorSharp docs/models/gemma4.md, "4.6 MoE", step 2):
// logits[t, e] = raw[t, e] / sqrt(mean_e raw[t, e]^2 + eps) * scale[e], in place,
// one warp per token; the mean of squares is summed in fp32 in a fixed order
// (lanes, then a shuffle tree).  scale == nullptr: all ones.
__global__ void moe_router_norm_kernel(float* __restrict__ logits, int m, int n_experts,
                                       const float* __restrict__ scale, float eps) {
  pdl_wait();  // the raw logits come from the previous grid
  pdl_launch_dependents();
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= m) return;
  float* row = logits + static_cast<size_t>(t) * n_experts;
  float ss = 0.f;
  for (int e = lane; e < n_experts; e += 32) ss = fmaf(row[e], row[e], ss);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float inv = rsqrtf(ss / static_cast<float>(n_experts) + eps);
  for (int e = lane; e < n_experts; e += 32) row[e] = row[e] * inv * (scale ? __ldg(scale + e) : 1.f);
}

// out[t, j] = bf16( sum_r probs[t, r] * d[t*top_k + r, j] + d[m*top_k + t, j] ), fixed order.
__global__ void moe_combine_kernel(const float* __restrict__ d, const float* __restrict__ probs, int m, int top_k,
                                   int cols, bool shared, uint16_t* __restrict__ out) {
  pdl_wait();  // d comes from the previous grid
  pdl_launch_dependents();
  const size_t total = static_cast<size_t>(m) * cols;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / cols), j_col = static_cast<int>(i - static_cast<size_t>(t) * cols);
    float acc = 0.f;
    // fixed slot order; the loads of 8 slots are issued before they are summed
    for (int r0 = 0; r0 < top_k; r0 += 8) {
      float pv[8], dv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = r0 + j;
        pv[j] = r < top_k ? __ldg(probs + t * top_k + r) : 0.f;
        dv[j] = r < top_k ? __ldg(d + static_cast<size_t>(t * top_k + r) * cols + j_col) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (r0 + j < top_k) acc = fmaf(pv[j], dv[j], acc);
    }
    if (shared) acc += __ldg(d + static_cast<size_t>(m * top_k + t) * cols + j_col);
    out[i] = f32_to_bf16_bits(acc);
  }
}

}  // namespace nvfp4
