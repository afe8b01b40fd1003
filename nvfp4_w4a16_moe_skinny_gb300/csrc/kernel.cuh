// The streaming kernel behind the dense skinny GEMM, the lm_head with its fused
// argmax, and the grouped MoE gate+up / down products.
//
// y[m, n] = sum_k w_hat[n, k] x[m, k] with NVFP4 weights (gemma-cuda-hybrid
// README, "Everything it has / Inference engine"): one kernel for every M<=16
// product, including the lm_heads (greedy argmax, "Headline numbers") and the
// expert-batched gate+up / down products of the MoE layer (TensorSharp
// docs/models/gemma4.md, "14. Optimization opportunities / Completed").
//
// Work decomposition.  A job is a list of *segments* (one matrix for the dense
// GEMM and the lm_head; the experts that received tokens, then the shared
// expert, for the MoE).  Each segment's matrix has `ng` 64-row groups and `kc`
// 64-column chunks; K may be cut into S slices of L chunks.  The *pieces*
// (segment, slice, group) are numbered segment-major, then slice, then group,
// and dealt to the grid in contiguous, balanced ranges (one CTA of 16 warps per
// SM).  A CTA walks its range in *runs* of one segment: it stages that
// segment's tokens over the K columns the run touches (one barrier), and deals
// the run's pieces to its warps round-robin.  A warp streams a piece's chunks
// through its own ring, accumulating 4 tiles x tokens in registers.
//
// Epilogue.  S == 1: the piece holds the whole dot product and is finished in
// registers.  S > 1: the warp stores its partial (already in output units) in
// the fixup buffer and takes a ticket on the group's counter; the last of the S
// slices to arrive sums the S partials in slice order and finishes the group.
// No thread ever spins on another CTA.
#pragma once

#include "stream.cuh"

namespace nvfp4 {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;

enum { kEpiStore = 0, kEpiArgmax = 1, kEpiGated = 2, kEpiRows = 3 };
constexpr int kSharedSeg = -1;  // segment of the always-on shared expert
constexpr int kDenseSeg = -2;   // the single segment of a dense job

struct Job {
  const uint8_t* w;       // matrix 0 of the (stacked) weight
  const float* gs;        // global scales, one per matrix
  const uint8_t* w_sh;    // shared-expert matrix (MoE) or nullptr
  const float* gs_sh;
  size_t mat_bytes;       // repacked bytes of one matrix
  int n, k;               // logical rows and columns of one matrix
  int ng, kc;             // 64-row groups, 64-column chunks
  int S, L;               // k-slices per group, chunks per slice
  const uint16_t* x;      // activations, rows of length k
  int m;                  // tokens
  int n_experts, top_k;   // MoE routing (n_experts == 0: dense job)
  const int* offsets;     // [n_experts + 1]
  const int* pairs;       // [m * top_k]
  int x_by_pair;          // MoE: 1 -> activation row = pair index (down); 0 -> token (gate_up)
  int has_shared;
  uint16_t* y;            // kEpiStore: y[tok * y_ld + row];  kEpiGated: h[pair * y_ld + i]
  int y_ld;
  float* yf;              // kEpiRows: d[pair * yf_ld + row]
  int yf_ld;
  float* fix;             // fixup partials (S > 1)
  unsigned* fix_cnt;      // one counter per (segment, group)
  float* am_val;          // kEpiArgmax: per-CTA partial results [grid][m]
  int* am_idx;
  unsigned* am_cnt;
  float* max_logit;
  int* argmax;
  int ns;                 // ring stages per warp
  int xs_chunks;          // capacity of the staged-activation buffer, in chunks
};

template <int MT, bool kMMA>
struct Acc {
  static constexpr int NT = (MT + 7) / 8;
  static constexpr int kPerLane = kMMA ? 4 * NT * 4 : 4 * MT * 2;
};

__host__ __device__ inline size_t stream_smem_bytes(bool mma, int slots, int xs_chunks, int ns, int n_experts) {
  const int nt = (slots + 7) / 8;
  const size_t ring = static_cast<size_t>(kWarps) * ns * kStageBytes;
  const size_t bars = static_cast<size_t>(kWarps) * ns * 8;
  const size_t xs = mma ? static_cast<size_t>(nt) * xs_chunks * kXFragChunkBytes
                        : static_cast<size_t>(slots) * xs_chunks * kXCoreChunkBytes;
  const size_t misc = 16 * 4 * 5 + kWarps * 16 * 8 + (static_cast<size_t>(n_experts) + 4) * 4 + 16;
  return ring + bars + xs + misc;
}

__device__ __forceinline__ bool better(float v, int r, float bv, int br) {
  return v > bv || (v == bv && r < br);
}

__device__ __forceinline__ float gelu_tanh(float z) {
  // 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))
  const float u = 0.7978845608028654f * fmaf(0.044715f * z, z * z, z);
  return 0.5f * z * (1.0f + tanhf(u));
}

template <int MT, bool kMMA, int kEpi>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(const Job p) {
  constexpr int NT = Acc<MT, kMMA>::NT;
  constexpr int SLOTS = kMMA ? NT * 8 : MT;
  constexpr int NACC = Acc<MT, kMMA>::kPerLane;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- shared memory carve-up
  const size_t ring_bytes = static_cast<size_t>(kWarps) * p.ns * kStageBytes;
  Ring ring{smem + static_cast<size_t>(warp) * p.ns * kStageBytes,
            reinterpret_cast<uint64_t*>(smem + ring_bytes) + warp * p.ns, p.ns};
  uint8_t* xs = smem + ring_bytes + static_cast<size_t>(kWarps) * p.ns * 8;
  const size_t xs_bytes = kMMA ? static_cast<size_t>(NT) * p.xs_chunks * kXFragChunkBytes
                               : static_cast<size_t>(SLOTS) * p.xs_chunks * kXCoreChunkBytes;
  int* sigma = reinterpret_cast<int*>(xs + xs_bytes);
  float* mul = reinterpret_cast<float*>(sigma + 16);
  int* slot_row = reinterpret_cast<int*>(mul + 16);
  int* slot_out = slot_row + 16;
  unsigned* s_amax = reinterpret_cast<unsigned*>(slot_out + 16);
  float* red_v = reinterpret_cast<float*>(s_amax + 16);
  int* red_i = reinterpret_cast<int*>(red_v + kWarps * 16);
  int* seg_list = red_i + kWarps * 16;   // [n_experts + 1]
  int* misc = seg_list + p.n_experts + 2;  // [0] = segment count, [1] = last-arrival flag

  // ---- segments
  if (p.n_experts == 0) {
    if (threadIdx.x == 0) seg_list[0] = kDenseSeg, misc[0] = 1;
  } else if (warp == 0) {
    int n = 0;
    for (int base = 0; base < p.n_experts; base += 32) {
      const int e = base + lane;
      const bool act = e < p.n_experts && __ldg(p.offsets + e + 1) > __ldg(p.offsets + e);
      const uint32_t mask = __ballot_sync(0xffffffffu, act);
      if (act) seg_list[n + __popc(mask & ((1u << lane) - 1u))] = e;
      n += __popc(mask);
    }
    if (lane == 0) {
      if (p.has_shared) seg_list[n++] = kSharedSeg;
      misc[0] = n;
    }
  }
  __syncthreads();
  const int n_seg = misc[0];
  const int per_seg = p.S * p.ng;  // pieces per segment
  const long long n_pieces = static_cast<long long>(n_seg) * per_seg;
  const int p0 = static_cast<int>(n_pieces * blockIdx.x / gridDim.x);
  const int p1 = static_cast<int>(n_pieces * (blockIdx.x + 1) / gridDim.x);

  // runs: consecutive pieces of one segment
  const int seg0 = per_seg ? p0 / per_seg : 0;
  const int n_runs = (p1 > p0) ? (p1 - 1) / per_seg - seg0 + 1 : 0;
  auto run_lo = [&](int r) { return max(p0, (seg0 + r) * per_seg); };
  auto run_hi = [&](int r) { return min(p1, (seg0 + r + 1) * per_seg); };
  auto run_units = [&](int r) {
    const int len = run_hi(r) - run_lo(r);
    return len > warp ? (len - warp + kWarps - 1) / kWarps : 0;
  };
  auto matrix_of = [&](int seg) -> const uint8_t* {
    const int e = seg_list[seg];
    if (e == kSharedSeg) return p.w_sh;
    if (e == kDenseSeg) return p.w;
    return p.w + static_cast<size_t>(e) * p.mat_bytes;
  };
  // piece -> (slice, group); chunks of slice s are [s*L, min(kc, (s+1)*L))
  auto slice_of = [&](int piece, int seg) { return (piece - seg * per_seg) / p.ng; };
  auto group_of = [&](int piece, int seg) { return (piece - seg * per_seg) % p.ng; };
  auto slice_len = [&](int s) { return min(p.kc, (s + 1) * p.L) - s * p.L; };

  // ---- producer (lane 0): cursor over this warp's pieces; chunk addresses are
  // recomputed only at piece boundaries (a piece's chunks are contiguous)
  int pr = 0, pu = 0;             // run, unit of the next piece to open
  const uint8_t* pptr = nullptr;  // next chunk to copy
  int prem = 0;                   // chunks left in the open piece
  const uint64_t policy = l2_evict_first_policy();
  auto issue_next = [&](int stage) {
    if (prem == 0) {
      while (pr < n_runs && pu >= run_units(pr)) pu = 0, ++pr;
      if (pr >= n_runs) return;
      const int seg = seg0 + pr;
      const int piece = run_lo(pr) + warp + pu * kWarps;
      const int sl = slice_of(piece, seg), grp = group_of(piece, seg);
      pptr = matrix_of(seg) + (static_cast<size_t>(grp) * p.kc + sl * p.L) * kStageBytes;
      prem = slice_len(sl);
      ++pu;
    }
    ring_issue(ring, stage, pptr, policy);
    pptr += kStageBytes;
    --prem;
  };
  ring_init(ring, lane);
  if (lane == 0)
    for (int st = 0; st < p.ns; ++st) issue_next(st);

  const int g = lane >> 2, t4 = lane & 3;
  const CoreLane cl(lane);
  float acc[kMMA ? 4 : 4][kMMA ? NT : MT][kMMA ? 4 : 2];
  constexpr int NBEST = kMMA ? NT * 2 : MT;
  float bv[NBEST];
  int bi[NBEST];
#pragma unroll
  for (int i = 0; i < NBEST; ++i) bv[i] = -INFINITY, bi[i] = 0x7FFFFFFF;

  // Finish a group whose full dot products are in `acc` (output units, i.e. already
  // multiplied by mul).  grp = 64-row group within the segment.
  auto finish = [&](int grp, int e) {
    if constexpr (!kMMA) {
      // CUDA-core partials are per 16-column group q: sum over the 4 lanes of a row pair
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int mm = 0; mm < MT; ++mm)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float v = acc[r][mm][h];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            acc[r][mm][h] = v;
          }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int rb = grp * 4 + r;  // 16-row block within the matrix
#pragma unroll
      for (int a = 0; a < (kMMA ? NT : MT); ++a)
#pragma unroll
        for (int i = 0; i < (kMMA ? 4 : 2); ++i) {
          const int hrow = kMMA ? (i >> 1) : i;                        // 0: row g, 1: row g+8
          const int slot = kMMA ? a * 8 + 2 * t4 + (i & 1) : a;
          const float v = acc[r][a][i];
          if constexpr (kEpi == kEpiStore) {
            const int row = rb * 16 + g + 8 * hrow;
            if ((kMMA || t4 == 0) && slot < p.m && row < p.n)
              p.y[static_cast<size_t>(slot) * p.y_ld + row] = f32_to_bf16_bits(v);
          } else if constexpr (kEpi == kEpiRows) {
            const int row = rb * 16 + g + 8 * hrow;
            const int out = slot_out[slot];
            if ((kMMA || t4 == 0) && out >= 0 && row < p.n) p.yf[static_cast<size_t>(out) * p.yf_ld + row] = v;
          } else if constexpr (kEpi == kEpiArgmax) {
            const int row = rb * 16 + g + 8 * hrow;
            const int b = kMMA ? a * 2 + (i & 1) : a;
            if (row < p.n && better(v, row, bv[b], bi[b])) bv[b] = v, bi[b] = row;
          } else {  // kEpiGated: rows g = gate i, g+8 = up i of block rb, i = rb*8 + g
            if (hrow == 0) {
              const float gate = v, up = acc[r][a][kMMA ? i + 2 : 1];
              const int out = slot_out[slot];
              if ((kMMA || t4 == 0) && out >= 0)
                p.y[static_cast<size_t>(out) * p.y_ld + rb * 8 + g] = f32_to_bf16_bits(gelu_tanh(gate) * up);
            }
          }
        }
    }
    (void)e;
  };

  int st = 0;            // ring stage of the next chunk
  uint32_t ph = 0;       // its mbarrier parity
  bool failed = false;   // a copy did not complete in time
  // every warp runs every iteration of this loop (its barriers are CTA-wide); a
  // warp whose copy timed out only skips its own chunks
  for (int r = 0; r < n_runs; ++r) {
    const int seg = seg0 + r;
    const int e = seg_list[seg];
    const int lo = run_lo(r), hi = run_hi(r);
    const int s_lo = slice_of(lo, seg), s_hi = slice_of(hi - 1, seg);
    const int kc_lo = s_lo * p.L, kc_hi = min(p.kc, (s_hi + 1) * p.L);
    // ---- stage this run's tokens over columns [64 kc_lo, 64 kc_hi)
    __syncthreads();
    if (threadIdx.x < 16) {
      const int j = threadIdx.x;
      int row = -1, out = -1;
      if (e == kDenseSeg) {
        if (j < p.m) row = out = j;
      } else if (e == kSharedSeg) {
        if (j < p.m) out = p.m * p.top_k + j, row = p.x_by_pair ? out : j;
      } else {
        const int o = __ldg(p.offsets + e), cnt = __ldg(p.offsets + e + 1) - o;
        if (j < cnt) {
          out = __ldg(p.pairs + o + j);
          row = p.x_by_pair ? out : out / p.top_k;
        }
      }
      slot_row[j] = j < SLOTS ? row : -1;
      slot_out[j] = j < SLOTS ? out : -1;
    }
    __syncthreads();
    auto tok_row = [&](int slot) -> int { return slot_row[slot]; };
    stage_tokens<kMMA, SLOTS>(p.x, p.k, kc_lo * kTileK, kc_hi - kc_lo, tok_row, s_amax, sigma, xs);
    if (threadIdx.x < SLOTS) {
      const float gsc = (e == kSharedSeg) ? __ldg(p.gs_sh) : (e == kDenseSeg ? __ldg(p.gs) : __ldg(p.gs + e));
      mul[threadIdx.x] = gsc * exp2i(8 - sigma[threadIdx.x]);
    }
    __syncthreads();

    const int units = run_units(r);
    for (int u = 0; u < units && !failed; ++u) {
      const int piece = lo + warp + u * kWarps;
      const int s = slice_of(piece, seg), grp = group_of(piece, seg);
      const int nch = slice_len(s);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < (kMMA ? NT : MT); ++b)
#pragma unroll
          for (int i = 0; i < (kMMA ? 4 : 2); ++i) acc[a][b][i] = 0.f;
      const uint8_t* xchunk = xs + static_cast<size_t>(s * p.L - kc_lo) * (kMMA ? NT * kXFragChunkBytes : MT * kXCoreChunkBytes);
      for (int c = 0; c < nch; ++c) {
        if (!mbar_wait_warp(&ring.bar[st], ph)) {
          failed = true;
          break;
        }
        const uint8_t* stage = ring.buf + st * kStageBytes;
        if constexpr (kMMA) {
          mma_chunk<NT>(stage, xchunk, lane, acc);
          xchunk += NT * kXFragChunkBytes;
        } else {
          core_chunk<MT>(stage, xchunk, cl, acc);
          xchunk += MT * kXCoreChunkBytes;
        }
        __syncwarp();
        if (lane == 0) {
          fence_proxy_async_smem();
          issue_next(st);
        }
        if (++st == p.ns) st = 0, ph ^= 1u;
      }
      if (failed) break;
      // ---- to output units
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < (kMMA ? NT : MT); ++b)
#pragma unroll
          for (int i = 0; i < (kMMA ? 4 : 2); ++i)
            acc[a][b][i] *= mul[kMMA ? b * 8 + 2 * t4 + (i & 1) : b];
      if (kEpi == kEpiArgmax || p.S == 1) {  // the lm_head never splits K
        finish(grp, e);
      } else if constexpr (kEpi != kEpiArgmax) {
        // ---- k-split: store the partial, take a ticket; the last slice sums all S in order
        const size_t gglob = static_cast<size_t>(seg) * p.ng + grp;
        float* mine = p.fix + ((gglob * p.S + s) * 32 + lane) * NACC;
        constexpr int B = kMMA ? NT : MT, C = kMMA ? 4 : 2;
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < B; ++b) {
            float* dst = mine + (a * B + b) * C;
            if constexpr (kMMA)
              __stcg(reinterpret_cast<float4*>(dst), make_float4(acc[a][b][0], acc[a][b][1], acc[a][b][2], acc[a][b][3]));
            else
              __stcg(reinterpret_cast<float2*>(dst), make_float2(acc[a][b][0], acc[a][b][1]));
          }
        __threadfence();
        __syncwarp();
        unsigned ticket = 0;
        if (lane == 0) ticket = atomicAdd(&p.fix_cnt[gglob], 1u);
        ticket = __shfl_sync(0xffffffffu, ticket, 0);
        if (ticket == static_cast<unsigned>(p.S - 1)) {
          if (lane == 0) atomicExch(&p.fix_cnt[gglob], 0u);
          __threadfence();
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < B; ++b)
#pragma unroll
              for (int i = 0; i < C; ++i) acc[a][b][i] = 0.f;
          // slices in fixed order, up to kBatch slices' loads in flight at once
          constexpr int kBatch = (kMMA && NT == 2) ? 1 : 2;  // registers: acc + kBatch slices
          for (int s0 = 0; s0 < p.S; s0 += kBatch) {
            constexpr int V = kMMA ? 4 : 2;
            float buf[kBatch][4][B][V];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
              if (s0 + j < p.S) {
                const float* src = p.fix + ((gglob * p.S + s0 + j) * 32 + lane) * NACC;
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                  for (int b = 0; b < B; ++b) {
                    const float* sp = src + (a * B + b) * C;
                    if constexpr (kMMA) {
                      const float4 f = __ldcg(reinterpret_cast<const float4*>(sp));
                      buf[j][a][b][0] = f.x, buf[j][a][b][1] = f.y, buf[j][a][b][2 % V] = f.z, buf[j][a][b][3 % V] = f.w;
                    } else {
                      const float2 f = __ldcg(reinterpret_cast<const float2*>(sp));
                      buf[j][a][b][0] = f.x, buf[j][a][b][1 % V] = f.y;
                    }
                  }
              }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
              if (s0 + j < p.S) {
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                  for (int b = 0; b < B; ++b)
#pragma unroll
                    for (int i = 0; i < C; ++i) acc[a][b][i] += buf[j][a][b][i];
              }
          }
          finish(grp, e);
        }
      }
    }
  }
  if (failed) {
    // a copy did not complete in time: wait (bounded) for the copies this warp
    // may still have in flight so none lands after the CTA exits, then give up
    for (int i = 1; i < p.ns; ++i) {
      if (++st == p.ns) st = 0, ph ^= 1u;
      (void)mbar_wait_warp(&ring.bar[st], ph);
    }
  }

  if constexpr (kEpi == kEpiArgmax) {
    // ---- lanes -> warp (ties to the lower row)
#pragma unroll
    for (int b = 0; b < NBEST; ++b) {
      float v = bv[b];
      int rw = bi[b];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, off);
        const int orow = __shfl_xor_sync(0xffffffffu, rw, off);
        if (better(ov, orow, v, rw)) v = ov, rw = orow;
      }
      const int slot = kMMA ? (b >> 1) * 8 + 2 * t4 + (b & 1) : b;
      if (kMMA ? g == 0 : lane == 0) red_v[warp * 16 + slot] = v, red_i[warp * 16 + slot] = rw;
    }
    __syncthreads();
    // ---- warps -> CTA, fixed order
    if (threadIdx.x < p.m) {
      const int tok = threadIdx.x;
      float v = -INFINITY;
      int rw = 0x7FFFFFFF;
      for (int w = 0; w < kWarps; ++w)
        if (better(red_v[w * 16 + tok], red_i[w * 16 + tok], v, rw)) v = red_v[w * 16 + tok], rw = red_i[w * 16 + tok];
      p.am_val[static_cast<size_t>(blockIdx.x) * p.m + tok] = v;
      p.am_idx[static_cast<size_t>(blockIdx.x) * p.m + tok] = rw;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned ticket = atomicAdd(p.am_cnt, 1u);
      const int last = ticket == gridDim.x - 1;
      if (last) atomicExch(p.am_cnt, 0u);
      misc[1] = last;
    }
    __syncthreads();
    if (misc[1] && threadIdx.x < p.m) {
      __threadfence();
      const int tok = threadIdx.x;
      float v = -INFINITY;
      int rw = 0x7FFFFFFF;
      for (unsigned b = 0; b < gridDim.x; ++b) {
        const float ov = __ldcg(p.am_val + static_cast<size_t>(b) * p.m + tok);
        const int orow = __ldcg(p.am_idx + static_cast<size_t>(b) * p.m + tok);
        if (better(ov, orow, v, rw)) v = ov, rw = orow;
      }
      p.max_logit[tok] = v;
      p.argmax[tok] = rw;
    }
  }
}

}  // namespace nvfp4
