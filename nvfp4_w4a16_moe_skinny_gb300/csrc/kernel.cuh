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
// expert, for the MoE).  Each segment's matrix has `ng` 64-row groups of four
// 16-row tiles and `kc` 64-column chunks; K may be cut into S slices of L
// chunks.  A *unit* is (segment, slice, group); units are numbered
// segment-major, then slice, then group, and dealt to the grid in contiguous,
// balanced ranges (one CTA of 16 warps per SM).  A CTA with at least 16 units
// deals them whole, round-robin over its warps (the SM's issue slots, not the
// warps, are then the limit, and whole units keep every copy four tiles wide);
// a CTA with fewer deals their tiles as contiguous ranges, so every warp has
// work.  A *piece* is one warp's share of one unit: 1 to 4 adjacent tiles over
// the unit's K slice, streamed as TMA boxes of 4 tiles x 1 chunk, 3 x 1, 2 x 2
// or 1 x 4.
//
// Each CTA stages its activations once (the token rows over the columns its
// units touch, or, for the down product, the gate+up outputs of its experts'
// pairs), before any piece starts.
//
// Epilogue.  S == 1: the piece holds whole dot products and is finished in
// registers.  S > 1: per tile, the warp stores its partial (already in output
// units) in the fixup buffer and takes a ticket on the tile's counter; the
// last of the S slices to arrive sums the S partials in slice order and
// finishes the tile.  No thread ever spins on another CTA.
//
// Launch overlap.  Weights never depend on the previous kernel, so every warp
// issues its first copies, then the CTA waits for the previous grid in the stream
// (griddepcontrol.wait) before it reads activations, routing or workspace, and
// only then lets the next grid start.  Outputs of the grid before the previous
// one are therefore complete when a CTA starts: the down product reads the
// routing before its wait.
#pragma once

#include <type_traits>

#include "stream.cuh"

namespace nvfp4 {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxCtaSegs = 8;                 // segments whose units one CTA may hold
constexpr int kMaxStagedRows = kMaxCtaSegs * 16;

// kEpiSample: the argmax of logit / T + Gumbel noise (temperature sampling)
enum { kEpiStore = 0, kEpiArgmax = 1, kEpiGated = 2, kEpiRows = 3, kEpiSample = 4 };
constexpr int kSharedSeg = -1;  // segment of the always-on shared expert
constexpr int kDenseSeg = -2;   // the single segment of a dense job

constexpr unsigned kErrPlan = 2u;  // a CTA's share exceeded the launch plan (g_device_error bit 1)

struct Job {
  const uint8_t* w;       // the (stacked) weight: matrix e, group G, chunk c at ((e*ng + G)*kc + c)*2304
  const float* gs;        // global scales, one per matrix
  const uint8_t* w_sh;    // shared-expert matrix (MoE) or nullptr
  const float* gs_sh;     // global scale of the shared expert (MoE) or nullptr
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
  int routing_ready;      // 1: the routing is complete before this grid starts (read before the wait)
  uint16_t* y;            // kEpiStore: y[tok * y_ld + row];  kEpiGated: h[pair * y_ld + i]
  int y_ld;
  float* yf;              // kEpiRows: d[pair * yf_ld + row]; kEpiStore: fp32 y if set (else bf16 y)
  int yf_ld;
  float* fix;             // fixup partials (S > 1)
  unsigned* fix_cnt;      // one counter per (segment, group, tile)
  unsigned long long* am_key;  // kEpiArgmax / kEpiSample: per-token packed (value, row) maxima [m]
  unsigned* am_cnt;
  float* max_logit;
  int* argmax;
  int ns;                 // ring stages per warp
  int npre;               // ring stages each warp fills before waiting for the previous grid
  int slice_ctas;         // single-segment job: CTA ranges aligned to K slices (see DecodeDeal)
  int xs_chunks;          // staged-activation capacity: chunks per row
  int xs_rows;            // staged-activation capacity: rows (plus the zero row)
  int max_cta_segs;       // segments one CTA may touch (<= kMaxCtaSegs)
  int max_segs;           // prefill kernel: capacity of the segment list
  float inv_temp;         // kEpiSample: 1 / temperature
  uint32_t seed_lo, seed_hi;  // kEpiSample: the Philox key of this call's noise
  float softcap;          // kEpiArgmax / kEpiSample: cap of cap * tanh(logit / cap) (0: off)
  const uint8_t* xq;      // W4A4 (dense jobs): NVFP4 activation codes [m, k/2] instead of x ...
  const uint8_t* xq_sc;   //   ... their E4M3 scales [m, k/16]
  const float* xq_g;      //   ... and per-row global scales [m]
};

__host__ __device__ inline size_t stream_table_bytes(int n_experts) {
  return static_cast<size_t>(4) * (kMaxStagedRows + (kMaxStagedRows + 1) + kMaxCtaSegs * 16 * 3 +
                                   kWarps * 16 * 2 + kWarps * 8 + n_experts + 2 + 4 + n_experts + 1);
}

__host__ __device__ inline size_t stream_smem_bytes(int xs_rows, int xs_chunks, int ns, int n_experts) {
  const size_t ring = static_cast<size_t>(kWarps) * ns * kStageBytes;
  const size_t bars = static_cast<size_t>(kWarps) * ns * 8;
  const size_t xs = static_cast<size_t>(xs_rows + 1) * (static_cast<size_t>(xs_chunks) * kXChunkBytes + 16);
  return ring + bars + xs + stream_table_bytes(n_experts);
}

// Whole-unit dealing for a CTA of nu units: the busiest warp then streams
// ceil(nu/16) units of four tiles, against ceil(4nu/16) split tiles otherwise.
__host__ __device__ inline bool deal_whole(long long nu) {
  const long long whole = (nu + kWarps - 1) / kWarps * 4 * 100;
  const long long split = (4 * nu + kWarps - 1) / kWarps * 115;
  return whole <= split;
}

// Units a CTA of nu units deals whole (round-robin over its warps); the rest
// are dealt as contiguous tile ranges.  All whole when the busiest warp's cost
// (whole tiles at 100, split tiles at 115) is no higher than all split; else
// all split.  (Whole full rounds with the remainder split balance the warps
// better but measured slower at M = 15: the SM's issue slots, not the busiest
// warp, bound the tile loop there, and split tiles cost more instructions.)
__host__ __device__ inline int whole_units(int nu) { return deal_whole(nu) ? nu : 0; }

__host__ __device__ constexpr int imin_(int a, int b) { return a < b ? a : b; }

// One warp's share of one unit: 1 to 4 adjacent tiles of (segment, K slice,
// 64-row group).
struct Piece {
  int seg, s, grp, t0, tn;
};

// The decode kernel's work decomposition, used by the kernel and by the
// host-side plan check (nvfp4_plan_check), so both walk the same code.  Units
// are (segment, slice, group), numbered segment-major, then slice, then group.
// CTA b owns the contiguous units [u0, u1): a balanced share of all units, or,
// for a single-segment job planned with slice_ctas (the grid a multiple of S),
// a balanced share of the groups of slice b / (grid / S), so that it stages one
// slice of K.  The CTA deals whole_units(nu) of its units whole, round-robin
// over its warps, and the rest as contiguous tile ranges.
struct DecodeDeal {
  int n_seg, S, L, kc, ng, grid, slice_ctas;
  __host__ __device__ int per_seg() const { return S * ng; }
  __host__ __device__ void cta_range(int b, int& u0, int& u1) const {
    if (slice_ctas && n_seg == 1 && S > 1 && grid % S == 0) {
      const int cps = grid / S, s = b / cps, j = b % cps;
      u0 = s * ng + static_cast<int>(static_cast<long long>(ng) * j / cps);
      u1 = s * ng + static_cast<int>(static_cast<long long>(ng) * (j + 1) / cps);
      return;
    }
    const long long n_units = static_cast<long long>(n_seg) * per_seg();
    u0 = static_cast<int>(n_units * b / grid);
    u1 = static_cast<int>(n_units * (b + 1) / grid);
  }
  __host__ __device__ int slice_len(int s) const { return imin_(kc, (s + 1) * L) - s * L; }
  // the CTA's first segment, segment count and staged chunks [c_lo, c_hi)
  __host__ __device__ void span(int u0, int u1, int& cseg0, int& nsc, int& c_lo, int& c_hi) const {
    const int nu = u1 - u0;
    cseg0 = nu > 0 ? u0 / per_seg() : 0;
    nsc = nu > 0 ? (u1 - 1) / per_seg() - cseg0 + 1 : 0;
    c_lo = 0, c_hi = nu > 0 ? kc : 0;
    if (nsc == 1) {
      c_lo = ((u0 - cseg0 * per_seg()) / ng) * L;
      c_hi = imin_(kc, ((u1 - 1 - cseg0 * per_seg()) / ng + 1) * L);
    }
  }
  // warp w's pieces of the CTA's nu units starting at u0: its whole units (units
  // w, w+16, ... of the first whole_units(nu)), then its contiguous tile range of
  // the remaining units
  __host__ __device__ int n_pieces(int nu, int w) const {
    const int nw = whole_units(nu), rest = nu - nw;
    const int whole = nw > w ? (nw - w + kWarps - 1) / kWarps : 0;
    const int T0 = (4 * rest * w) / kWarps, T1 = (4 * rest * (w + 1)) / kWarps;
    return whole + (T1 > T0 ? ((T1 - 1) >> 2) - (T0 >> 2) + 1 : 0);
  }
  __host__ __device__ Piece piece(int u0, int nu, int w, int k) const {
    const int nw = whole_units(nu), rest = nu - nw;
    const int whole = nw > w ? (nw - w + kWarps - 1) / kWarps : 0;
    int unit, t0, tn;
    if (k < whole) {
      unit = u0 + k * kWarps + w, t0 = 0, tn = 4;
    } else {
      const int kk = k - whole;
      const int T0 = (4 * rest * w) / kWarps, T1 = (4 * rest * (w + 1)) / kWarps;
      const int start = kk == 0 ? T0 : ((T0 >> 2) + kk) << 2;
      const int end = imin_(T1, ((T0 >> 2) + kk + 1) << 2);
      unit = u0 + nw + (start >> 2), t0 = start & 3, tn = end - start;
    }
    Piece pc;
    pc.seg = unit / per_seg();
    const int r = unit - pc.seg * per_seg();
    pc.s = r / ng;
    pc.grp = r - pc.s * ng;
    pc.t0 = t0, pc.tn = tn;
    return pc;
  }
};

__device__ __forceinline__ bool better(float v, int r, float bv, int br) {
  return v > bv || (v == bv && r < br);
}

// (value, row) as one unsigned 64-bit key whose order is `better`'s: the fp32 bits
// made order-preserving as unsigned (sign bit flipped for non-negative values,
// all bits inverted for negative ones) above the inverted row.  Never 0 for a
// finite or infinite value, so 0 is below every key.
__device__ __forceinline__ unsigned long long pack_value_row(float v, int row) {
  const uint32_t u = __float_as_uint(v);
  const uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(k) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(row));
}
__device__ __forceinline__ float unpack_value(unsigned long long key) {
  const uint32_t k = static_cast<uint32_t>(key >> 32);
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ int unpack_row(unsigned long long key) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key));
}

__device__ __forceinline__ float gelu_tanh(float z) {
  // 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))
  const float u = 0.7978845608028654f * fmaf(0.044715f * z, z * z, z);
  return 0.5f * z * (1.0f + tanhf(u));
}

template <int MT, bool kMMA, int kEpi>
__global__ void __launch_bounds__(kThreads, 1)
    stream_kernel(const __grid_constant__ Job p, const __grid_constant__ WeightMaps maps) {
  constexpr int NT = (MT + 7) / 8;
  constexpr int NA = kMMA ? NT : MT;   // accumulator columns per tile
  constexpr int NI = kMMA ? 4 : 2;     // floats per accumulator column
  constexpr int V = NA * NI;           // accumulator floats per lane and tile
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;

  // ---- shared memory carve-up: warp w's stages at smem + w*ns*2304, then one
  // mbarrier per stage, the staged activations and the tables
  const int ns = p.ns;
  const size_t ring_bytes = static_cast<size_t>(kWarps) * ns * kStageBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + ring_bytes) + warp * ns;  // this warp's barriers
  uint8_t* xs = smem + ring_bytes + static_cast<size_t>(kWarps) * ns * 8;
  const size_t xs_bytes = static_cast<size_t>(p.xs_rows + 1) * (static_cast<size_t>(p.xs_chunks) * kXChunkBytes + 16);
  int* row_src = reinterpret_cast<int*>(xs + xs_bytes);                      // [kMaxStagedRows]
  int* sigma = row_src + kMaxStagedRows;                                     // [kMaxStagedRows + 1]
  int* slot_row = sigma + kMaxStagedRows + 1;                                // [kMaxCtaSegs * 16]
  int* slot_out = slot_row + kMaxCtaSegs * 16;
  float* mul = reinterpret_cast<float*>(slot_out + kMaxCtaSegs * 16);
  float* red_v = mul + kMaxCtaSegs * 16;                                     // [kWarps * 16]
  int* red_i = reinterpret_cast<int*>(red_v + kWarps * 16);
  int* cur = red_i + kWarps * 16 + warp * 8;                                 // [kWarps * 8] box cursors
  int* seg_list = red_i + kWarps * 16 + kWarps * 8;                          // [n_experts + 2]
  int* misc = seg_list + p.n_experts + 2;  // [0] segments, [1] last-arrival flag, [2] staged rows
  int* s_off = misc + 4;                   // [n_experts + 1] the expert offsets (MoE)

  if (lane == 0) {
    for (int s = 0; s < ns; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // ---- segments: the dense matrix, or the experts that received pairs, then the shared expert
  const bool dense = p.n_experts == 0;
  const bool early = dense || p.routing_ready;
  if (!early) pdl_wait();
  if (dense) {
    if (threadIdx.x == 0) seg_list[0] = kDenseSeg, misc[0] = 1;
  } else {
    // the offsets go to shared memory in one round of loads (one per thread), then
    // warp 0 lists the experts that received pairs
    for (int e = threadIdx.x; e <= p.n_experts; e += blockDim.x) s_off[e] = __ldg(p.offsets + e);
    __syncthreads();
    if (warp == 0) {
      int n = 0;
      for (int base = 0; base < p.n_experts; base += 32) {
        const int e = base + lane;
        const bool act = e < p.n_experts && s_off[e + 1] > s_off[e];
        const uint32_t mask = __ballot_sync(0xffffffffu, act);
        if (act) seg_list[n + __popc(mask & ((1u << lane) - 1u))] = e;
        n += __popc(mask);
      }
      if (lane == 0) {
        if (p.has_shared) seg_list[n++] = kSharedSeg;
        misc[0] = n;
      }
    }
  }
  __syncthreads();
  const DecodeDeal dd{misc[0], p.S, p.L, p.kc, p.ng, static_cast<int>(gridDim.x), p.slice_ctas};
  int u0, u1;
  dd.cta_range(blockIdx.x, u0, u1);
  int nu = u1 - u0;
  // this CTA's segments and K columns (chunks [c_lo, c_hi))
  int cseg0, nsc, c_lo, c_hi;
  dd.span(u0, u1, cseg0, nsc, c_lo, c_hi);
  if (nsc > p.max_cta_segs || c_hi - c_lo > p.xs_chunks || (smem_addr(smem) & 127u)) {
    // the launch plan does not cover this CTA's share: record it and do no work
    if (threadIdx.x == 0) atomicOr(&g_device_error, kErrPlan);
    nu = 0;
  }
  const int nsc_used = nu > 0 ? nsc : 0;
  if (nu == 0) c_lo = c_hi = 0;  // nothing to stage

  // ---- warp w's pieces: whole units round-robin (warp w takes units w, w+16,
  // ...), or the units' tiles as contiguous ranges, whichever leaves the busiest
  // warp less work (a split tile costs ~1.15x a tile of a whole unit: its x
  // fragments and scale work are not shared by four tiles)
  const int n_pieces = dd.n_pieces(nu, warp);
  auto piece_at = [&](int k) -> Piece { return dd.piece(u0, nu, warp, k); };
  auto slice_len = [&](int s) { return dd.slice_len(s); };

  // ---- producer (lane 0): cursor over this warp's pieces.  A whole unit (four
  // tiles) is one bulk copy of 2,304 contiguous bytes per chunk, from a source
  // pointer held in registers; a piece of 1-3 tiles is ceil(chunks /
  // copy_chunks(tn)) TMA boxes, whose cursor lives in shared memory (lane 0's
  // only: [0] map index, tn-1 or +4 for the shared expert, [1] t0, [2] next
  // chunk, [3] group, [4] chunks per copy).  The last box may run past the slice
  // (those chunks are loaded, or zero-filled past K, and not used).
  int pk = 0;                      // next piece to open
  int prem = 0;                    // copies left in the open piece
  const uint8_t* psrc = nullptr;   // next bulk-copy source; nullptr: the piece uses TMA boxes
  const uint64_t policy = l2_evict_first_policy();
  uint8_t* ring = smem + static_cast<size_t>(warp) * ns * kStageBytes;
  const uint32_t ring_s = smem_addr(ring), bar_s = smem_addr(bar);
  auto issue_next = [&](int stage) {
    if (prem == 0) {
      if (pk >= n_pieces) return;
      const Piece pc = piece_at(pk++);
      const int e = seg_list[pc.seg];
      const int group = (e >= 0 ? e * p.ng : 0) + pc.grp;  // within the stack
      if (pc.tn == kChunkTiles) {
        prem = slice_len(pc.s);
        psrc = (e == kSharedSeg ? p.w_sh : p.w) + (static_cast<size_t>(group) * p.kc + pc.s * p.L) * kStageBytes;
      } else {
        const int step = copy_chunks(pc.tn);
        prem = (slice_len(pc.s) + step - 1) / step;
        psrc = nullptr;
        cur[0] = (pc.tn - 1) + (e == kSharedSeg ? 4 : 0);
        cur[1] = pc.t0;
        cur[2] = pc.s * p.L;
        cur[3] = group;
        cur[4] = step;
      }
    }
    const uint32_t b = bar_s + stage * 8, d = ring_s + stage * kStageBytes;
    if (psrc) {
      mbar_arrive_expect_tx_s(b, kStageBytes);
      bulk_g2s_s(d, psrc, kStageBytes, b, policy);
      psrc += kStageBytes;
    } else {
      const int mi = cur[0];
      mbar_arrive_expect_tx_s(b, static_cast<uint32_t>(((mi & 3) + 1) * cur[4]) * kTileBytes);
      tma_load_4d_s(d, mi < 4 ? &maps.w[mi] : &maps.sh[mi - 4], 0, cur[1], cur[2], cur[3], b, policy);
      cur[2] += cur[4];
    }
    --prem;
  };
  // only the first npre stages go out before the wait for the previous grid: the
  // activation loads after the wait then queue behind few weight copies, and the
  // rest of the ring follows them (issue_rest, called once the loads are issued)
  const int npre = min(ns, p.npre);
  if (lane == 0)
    for (int st = 0; st < npre; ++st) issue_next(st);
  bool rest_issued = false;
  auto issue_rest = [&]() {
    if (!rest_issued) {
      rest_issued = true;
      if (lane == 0)
        for (int st = npre; st < ns; ++st) issue_next(st);
    }
  };

  // ---- staged rows and the (segment, slot) tables: they depend on the routing
  // only, so a job whose routing is complete builds them before the wait
  const int stride = (c_hi - c_lo) * kXChunkBytes + 16;
  // staged rows of local segment i: the m tokens (dense, gate+up: one copy for
  // all segments) or, for the down product, the segment's pairs' rows
  auto seg_rows = [&](int i) {
    const int e = seg_list[cseg0 + i];
    return e < 0 ? p.m : min(p.m, s_off[e + 1] - s_off[e]);
  };
  int nrows = 0;
  if (!p.x_by_pair) {
    nrows = nsc_used ? p.m : 0;
    for (int j = threadIdx.x; j < nrows; j += blockDim.x) row_src[j] = j;
  } else {
    for (int i = 0; i < nsc_used; ++i) nrows += seg_rows(i);
  }
  if (threadIdx.x < nsc_used * 16) {
    const int i = threadIdx.x >> 4, j = threadIdx.x & 15;
    const int e = seg_list[cseg0 + i];
    int row = nrows, out = -1;  // empty slot: the zero row, no output
    if (e == kDenseSeg) {
      if (j < p.m) row = out = j;
    } else {
      // first staged row of segment i (down product: rows are per segment)
      int base = 0;
      if (p.x_by_pair)
        for (int ii = 0; ii < i; ++ii) base += seg_rows(ii);
      if (e == kSharedSeg) {
        if (j < p.m) out = p.m * p.top_k + j, row = p.x_by_pair ? base + j : j;
      } else {
        const int o = s_off[e], cnt = min(p.m, s_off[e + 1] - o);
        if (j < cnt) {
          out = __ldg(p.pairs + o + j);
          row = p.x_by_pair ? base + j : out / p.top_k;
        }
      }
      if (p.x_by_pair && row < nrows) row_src[row] = out;
    }
    slot_row[threadIdx.x] = row;
    slot_out[threadIdx.x] = out;
  }
  __syncthreads();
  if (early) pdl_wait();
  pdl_launch_dependents();

  if (p.xq)  // W4A4: the rows are NVFP4 already
    stage_rows_fp4<kMMA>(p.xq, p.xq_sc, p.k, c_lo * kTileK, c_hi - c_lo, nrows, row_src, sigma, xs, stride,
                         issue_rest);
  else
    stage_rows<kMMA>(p.x, p.k, c_lo * kTileK, c_hi - c_lo, nrows, row_src, sigma, xs, stride, issue_rest);
  if (threadIdx.x < nsc_used * 16) {
    const int e = seg_list[cseg0 + (threadIdx.x >> 4)];
    const float gsc = (e == kSharedSeg) ? __ldg(p.gs_sh) : (e == kDenseSeg ? __ldg(p.gs) : __ldg(p.gs + e));
    const int row = slot_row[threadIdx.x];
    // (W4A4, dense jobs: staged row j is token j, with its own global scale)
    mul[threadIdx.x] = row < nrows ? gsc * exp2i(8 - sigma[row]) * (p.xq_g ? __ldg(p.xq_g + row) : 1.f) : 0.f;
  }
  __syncthreads();

  const CoreLane cl(lane);
  const uint32_t xs_addr = smem_addr(xs);
  float acc[4][NA][NI];
  constexpr int NBEST = kMMA ? NT * 2 : MT;
  float bv[NBEST];
  int bi[NBEST];
#pragma unroll
  for (int i = 0; i < NBEST; ++i) bv[i] = -INFINITY, bi[i] = 0x7FFFFFFF;

  // Finish tile t (0..3) of group grp of local segment sl from a[] (output units).
  auto finish_tile = [&](int sl, int grp, int t, const float (&a)[NA][NI]) {
    const int rb = grp * 4 + t;  // 16-row block within the matrix
#pragma unroll
    for (int c = 0; c < NA; ++c)
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int hrow = kMMA ? (i >> 1) : i;  // 0: row g, 1: row g+8
        const int slot = kMMA ? c * 8 + 2 * t4 + (i & 1) : c;
        const float v = a[c][i];
        const int row = rb * 16 + g + 8 * hrow;
        if constexpr (kEpi == kEpiStore) {
          if ((kMMA || t4 == 0) && slot < p.m && row < p.n) {
            if (p.yf)  // fp32 output (the router logits)
              p.yf[static_cast<size_t>(slot) * p.yf_ld + row] = v;
            else
              p.y[static_cast<size_t>(slot) * p.y_ld + row] = f32_to_bf16_bits(v);
          }
        } else if constexpr (kEpi == kEpiRows) {
          const int out = slot_out[sl * 16 + slot];
          if ((kMMA || t4 == 0) && out >= 0 && row < p.n) p.yf[static_cast<size_t>(out) * p.yf_ld + row] = v;
        } else if constexpr (kEpi == kEpiArgmax || kEpi == kEpiSample) {
          const int b = kMMA ? c * 2 + (i & 1) : c;
          float key = v;  // the logit, or (sampling) logit / T + the Gumbel noise of (row, token)
          if (p.softcap > 0.f) key = p.softcap * tanhf(key / p.softcap);  // the final-logit softcap
          if constexpr (kEpi == kEpiSample)
            if (row < p.n && slot < p.m)
              key = fmaf(key, p.inv_temp, gumbel_from_bits(philox4x32_10_word0(row, slot, p.seed_lo, p.seed_hi)));
          if (key != key) key = -INFINITY;  // a NaN counts as -inf: the result is always a valid row
          if (row < p.n && better(key, row, bv[b], bi[b])) bv[b] = key, bi[b] = row;
        } else {  // kEpiGated: rows g = gate i, g+8 = up i of block rb, i = rb*8 + g
          if (hrow == 0) {
            const float up = a[c][kMMA ? i + 2 : 1];
            const int out = slot_out[sl * 16 + slot];
            if ((kMMA || t4 == 0) && out >= 0)
              p.y[static_cast<size_t>(out) * p.y_ld + rb * 8 + g] = f32_to_bf16_bits(gelu_tanh(v) * up);
          }
        }
      }
  };


  {
    // ---- stream the pieces through the ring
    const uint32_t ring_addr = smem_addr(ring);
    int st = 0;           // ring stage of the next copy
    uint32_t ph = 0;      // its mbarrier parity
    bool failed = false;  // a copy did not complete in time
    for (int k = 0; k < n_pieces && !failed; ++k) {
      const Piece pc = piece_at(k);
      const int sl = pc.seg - cseg0;
      const int kc0 = pc.s * p.L, nch = slice_len(pc.s);
      const uint32_t xbase = xs_addr + (kc0 - c_lo) * kXChunkBytes;
      uint32_t xr[NA];
#pragma unroll
      for (int c = 0; c < NA; ++c) {
        if constexpr (kMMA)
          xr[c] = xbase + slot_row[sl * 16 + c * 8 + g] * stride + t4 * 32;
        else
          xr[c] = xbase + slot_row[sl * 16 + c] * stride;
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < NA; ++c)
#pragma unroll
          for (int i = 0; i < NI; ++i) acc[a][c][i] = 0.f;
      // the piece's copies; copy j holds chunks j*step .. of the slice, each TN tiles
      // at stage + c*TN*576 (one loop per TN, chosen once per piece)
      auto stream_piece = [&](auto tn_c) {
        constexpr int TN = decltype(tn_c)::value;
        constexpr int kStep = copy_chunks(TN);
        int ch = 0;
        if constexpr (kStep == 1 && !kMMA) {
          // CUDA cores (one token, issue-bound): whole chunks two at a time -- both
          // stages' waits, both chunks, both refills -- halving the per-chunk
          // wait and refill work.  Only with 4+ stages, so that two stay in flight
          // while the pair is consumed.  (The tensor-core path measured slower so.)
          for (; ns >= 4 && ch + 1 < nch; ch += 2) {
            const int st1 = st + 1 == ns ? 0 : st + 1;
            const uint32_t ph1 = st + 1 == ns ? ph ^ 1u : ph;
            if (!mbar_wait_warp(&bar[st], ph)) {
              failed = true;
              return;
            }
            if (!mbar_wait_warp(&bar[st1], ph1)) {
              st = st1, ph = ph1;  // the stage that timed out
              failed = true;
              return;
            }
            core_chunk<MT, TN>(ring_addr + st * kStageBytes, xr, cl, acc);
#pragma unroll
            for (int c = 0; c < NA; ++c) xr[c] += kXChunkBytes;
            core_chunk<MT, TN>(ring_addr + st1 * kStageBytes, xr, cl, acc);
#pragma unroll
            for (int c = 0; c < NA; ++c) xr[c] += kXChunkBytes;
            __syncwarp();
            if (lane == 0) {
              fence_proxy_async_smem();  // this warp's reads of both stages before the next copies into them
              issue_next(st);
              issue_next(st1);
            }
            st = st1 + 1 == ns ? 0 : st1 + 1;
            ph = st1 + 1 == ns ? ph1 ^ 1u : ph1;
          }
        }
        for (; ch < nch; ch += kStep) {
          if (!mbar_wait_warp(&bar[st], ph)) {
            failed = true;
            return;
          }
          const uint32_t stage = ring_addr + st * kStageBytes;
          if constexpr (kStep == 1) {
            if constexpr (kMMA)
              mma_chunk<NT, TN>(stage, xr, lane, acc);
            else
              core_chunk<MT, TN>(stage, xr, cl, acc);
#pragma unroll
            for (int c = 0; c < NA; ++c) xr[c] += kXChunkBytes;
          } else {
            const int cnt = min(kStep, nch - ch);  // chunks of this copy inside the slice
            for (int cc = 0; cc < cnt; ++cc) {
              if constexpr (kMMA)
                mma_chunk<NT, TN>(stage + cc * TN * kTileBytes, xr, lane, acc);
              else
                core_chunk<MT, TN>(stage + cc * TN * kTileBytes, xr, cl, acc);
#pragma unroll
              for (int c = 0; c < NA; ++c) xr[c] += kXChunkBytes;
            }
          }
          __syncwarp();
          if (lane == 0) {
            fence_proxy_async_smem();  // this warp's reads of the stage before the next copy into it
            issue_next(st);
          }
          if (++st == ns) st = 0, ph ^= 1u;
        }
      };
      switch (pc.tn) {
        case 4: stream_piece(std::integral_constant<int, 4>{}); break;
        case 3: stream_piece(std::integral_constant<int, 3>{}); break;
        case 2: stream_piece(std::integral_constant<int, 2>{}); break;
        default: stream_piece(std::integral_constant<int, 1>{}); break;
      }
      if (failed) break;
      // ---- to output units (CUDA cores: first the sum over the 4 lanes of a row pair)
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        if (a >= pc.tn) break;
#pragma unroll
        for (int c = 0; c < NA; ++c)
#pragma unroll
          for (int i = 0; i < NI; ++i) {
            float v = acc[a][c][i];
            if constexpr (!kMMA) {
              v += __shfl_xor_sync(0xffffffffu, v, 1);
              v += __shfl_xor_sync(0xffffffffu, v, 2);
            }
            acc[a][c][i] = v * mul[sl * 16 + (kMMA ? c * 8 + 2 * t4 + (i & 1) : c)];
          }
      }
      if (kEpi == kEpiArgmax || kEpi == kEpiSample || p.S == 1) {  // the lm_head never splits K
#pragma unroll
        for (int a = 0; a < 4; ++a)
          if (a < pc.tn) finish_tile(sl, pc.grp, pc.t0 + a, acc[a]);
      } else if constexpr (kEpi != kEpiArgmax && kEpi != kEpiSample) {
        // ---- k-split: per tile, store the partial and take a ticket; the last of
        // the S slices sums all S partials in slice order and finishes the tile
        const size_t cell0 = (static_cast<size_t>(pc.seg) * p.ng + pc.grp) * 4 + pc.t0;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          if (a >= pc.tn) break;
          float* dst = p.fix + (((cell0 + a) * p.S + pc.s) * 32 + lane) * V;
#pragma unroll
          for (int c = 0; c < NA; ++c) {
            if constexpr (kMMA)
              __stcg(reinterpret_cast<float4*>(dst + c * 4), make_float4(acc[a][c][0], acc[a][c][1], acc[a][c][2], acc[a][c][3]));
            else
              __stcg(reinterpret_cast<float2*>(dst + c * 2), make_float2(acc[a][c][0], acc[a][c][1]));
          }
        }
        __threadfence();
        __syncwarp();
        unsigned last = 0;  // bit a: this warp completed tile t0 + a
        if (lane == 0) {
          unsigned tk[4];
#pragma unroll
          for (int a = 0; a < 4; ++a)
            if (a < pc.tn) tk[a] = atomicAdd(&p.fix_cnt[cell0 + a], 1u);
#pragma unroll
          for (int a = 0; a < 4; ++a)
            if (a < pc.tn && tk[a] == static_cast<unsigned>(p.S - 1)) {
              last |= 1u << a;
              atomicExch(&p.fix_cnt[cell0 + a], 0u);
            }
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) __threadfence();
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          if (!((last >> a) & 1u)) continue;
          float sum[NA][NI];
#pragma unroll
          for (int c = 0; c < NA; ++c)
#pragma unroll
            for (int i = 0; i < NI; ++i) sum[c][i] = 0.f;
          const float* src0 = p.fix + ((cell0 + a) * p.S * 32 + lane) * V;
          constexpr int kBatch = V >= 8 ? 2 : 8;  // slices in flight together (registers)
          for (int s0 = 0; s0 < p.S; s0 += kBatch) {
            float buf[kBatch][NA][NI];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
              if (s0 + j < p.S) {
                const float* src = src0 + static_cast<size_t>(s0 + j) * 32 * V;
#pragma unroll
                for (int c = 0; c < NA; ++c) {
                  if constexpr (kMMA) {
                    const float4 f = __ldcg(reinterpret_cast<const float4*>(src + c * 4));
                    buf[j][c][0] = f.x, buf[j][c][1] = f.y, buf[j][c][2 % NI] = f.z, buf[j][c][3 % NI] = f.w;
                  } else {
                    const float2 f = __ldcg(reinterpret_cast<const float2*>(src + c * 2));
                    buf[j][c][0] = f.x, buf[j][c][1 % NI] = f.y;
                  }
                }
              }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
              if (s0 + j < p.S) {
#pragma unroll
                for (int c = 0; c < NA; ++c)
#pragma unroll
                  for (int i = 0; i < NI; ++i) sum[c][i] += buf[j][c][i];
              }
          }
          finish_tile(sl, pc.grp, pc.t0 + a, sum);
        }
      }
    }
    if (failed) {
      // a copy did not complete in time: wait (bounded) for the copies this warp
      // may still have in flight so none lands after the CTA exits, then give up
      for (int i = 1; i < ns; ++i) {
        if (++st == ns) st = 0, ph ^= 1u;
        (void)mbar_wait_warp(&bar[st], ph);
      }
    }
  }

  if constexpr (kEpi == kEpiArgmax || kEpi == kEpiSample) {
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
    // ---- warps -> CTA, fixed order, then CTAs -> grid: one 64-bit atomic max per
    // token on (orderable value, inverted row), whose maximum is the largest value
    // and, among equal values, the lowest row: the result does not depend on the
    // order the CTAs arrive in.  The last CTA to arrive reads and resets the keys.
    if (threadIdx.x < p.m) {
      const int tok = threadIdx.x;
      float v = -INFINITY;
      int rw = 0x7FFFFFFF;
      for (int w = 0; w < kWarps; ++w)
        if (better(red_v[w * 16 + tok], red_i[w * 16 + tok], v, rw)) v = red_v[w * 16 + tok], rw = red_i[w * 16 + tok];
      if (rw != 0x7FFFFFFF) atomicMax(p.am_key + tok, pack_value_row(v, rw));
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
      const unsigned long long key = atomicExch(p.am_key + threadIdx.x, 0ull);
      p.max_logit[threadIdx.x] = unpack_value(key);
      p.argmax[threadIdx.x] = unpack_row(key);
    }
  }
}

}  // namespace nvfp4
