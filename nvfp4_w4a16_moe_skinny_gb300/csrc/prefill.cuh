// The grouped MoE gate+up and down products for a prefill chunk (m > 16 tokens).
//
// The same contraction as the decode path (TensorSharp docs/models/gemma4.md,
// "14. Optimization opportunities / Completed": expert-batched gate+up and down
// over the tokens routed to each expert), when an expert may receive more than
// 16 pairs.  Each expert's pairs are cut into blocks of at most 32, and each
// block is a *segment* of 32 token slots: every dequantized 16x64 NVFP4 weight
// tile feeds four 8-slot m16n8k16 MMA columns (f16 in, fp32 accumulation), so an
// expert's weights are streamed and dequantized once per 32 pairs.  The shared
// expert is cut the same way into blocks of 32 tokens.
//
// Work decomposition.  A unit is (segment, K slice, 64-row group, half): two
// 16-row tiles.  Units are numbered segment-major, then slice, group and half,
// and dealt to the grid in contiguous balanced ranges; a warp's share of a unit
// (a piece, 1-2 tiles) streams through the warp's own ring of TMA boxes.  A
// CTA's range crosses (segment, slice) blocks, each with its own 32 activation
// rows over its own columns, so the CTA walks its range one block at a time (a
// *run*): it stages the run's rows, deals the run's units to its warps, and
// moves on once every warp is done.  The weight copies run ahead across runs;
// only the staging waits.  Runs never span slices, so the staged rows cover one
// slice and K may be split (S > 1, with the decode path's fixup) when a slice
// of 32 rows of the whole K would not fit beside the rings.
#pragma once

#include "kernel.cuh"

namespace nvfp4 {

constexpr int kPrefillSlots = 32;  // activation rows of one segment (four 8-slot MMA columns)

// Tables after the staged rows (4-byte entries): row_src[32], sigma[33],
// slot_row[32], slot_out[32], mul[32], the warps' copy cursors [16 x 8], the
// segment list and the block of each segment [max_segs + 1 each], misc[4].
constexpr int kPrefillFixedEntries = 5 * kPrefillSlots + 1 + kWarps * 8;

__host__ __device__ inline size_t prefill_table_bytes(int max_segs) {
  return static_cast<size_t>(4) * (kPrefillFixedEntries + 2 * (static_cast<size_t>(max_segs) + 1) + 4);
}

__host__ __device__ inline size_t prefill_smem_bytes(int xs_chunks, int ns, int max_segs) {
  const size_t ring = static_cast<size_t>(kWarps) * ns * kStageBytes;
  const size_t bars = static_cast<size_t>(kWarps) * ns * 8;
  const size_t xs = static_cast<size_t>(kPrefillSlots + 1) * (static_cast<size_t>(xs_chunks) * kXChunkBytes + 16);
  return ring + bars + xs + prefill_table_bytes(max_segs);
}

// The prefill kernel's work decomposition, used by the kernel and by the
// host-side plan check (nvfp4_plan_check).  A unit is (segment, K slice, 64-row
// group, half): two 16-row tiles.  CTA b owns [n_units*b/grid,
// n_units*(b+1)/grid); run r is its units of (segment, slice) block b0 + r; in a
// run, warp w takes whole units w, w+16, ... or the units' tiles as contiguous
// ranges, whichever leaves the busiest warp less work.
struct PrefillDeal {
  int n_seg, S, L, kc, ng, grid;
  __host__ __device__ int upg() const { return 2 * ng; }
  __host__ __device__ int per_seg() const { return S * upg(); }
  __host__ __device__ void cta_range(int b, int& u0, int& u1) const {
    const long long n_units = static_cast<long long>(n_seg) * per_seg();
    u0 = static_cast<int>(n_units * b / grid);
    u1 = static_cast<int>(n_units * (b + 1) / grid);
  }
  __host__ __device__ int n_runs(int u0, int u1) const { return u1 > u0 ? (u1 - 1) / upg() - u0 / upg() + 1 : 0; }
  __host__ __device__ int run_lo(int u0, int r) const { const int b = u0 / upg() + r; return b * upg() > u0 ? b * upg() : u0; }
  __host__ __device__ int run_hi(int u0, int u1, int r) const {
    const int e = (u0 / upg() + r + 1) * upg();
    return e < u1 ? e : u1;
  }
  __host__ __device__ int run_seg(int u0, int r) const { return (u0 / upg() + r) / S; }
  __host__ __device__ int run_slice(int u0, int r) const { return (u0 / upg() + r) - run_seg(u0, r) * S; }
  __host__ __device__ int slice_len(int s) const { return imin_(kc, (s + 1) * L) - s * L; }
  __host__ __device__ static bool whole(int nu) {
    return (nu + kWarps - 1) / kWarps * 2 * 100 <= (2 * nu + kWarps - 1) / kWarps * 115;
  }
  __host__ __device__ int n_pieces(int nu, int w) const {
    if (whole(nu)) return (nu - w + kWarps - 1) / kWarps;
    const int T0 = (2 * nu * w) / kWarps, T1 = (2 * nu * (w + 1)) / kWarps;
    return T1 > T0 ? ((T1 - 1) >> 1) - (T0 >> 1) + 1 : 0;
  }
  // piece k of warp w over the run's units [lo, lo + nu); t0 is the first tile (0..3) of the group
  __host__ __device__ Piece piece(int lo, int nu, int w, int k) const {
    int unit, t0, tn;
    if (whole(nu)) {
      unit = lo + k * kWarps + w, t0 = 0, tn = 2;
    } else {
      const int T0 = (2 * nu * w) / kWarps, T1 = (2 * nu * (w + 1)) / kWarps;
      const int start = k == 0 ? T0 : ((T0 >> 1) + k) << 1;
      const int end = imin_(T1, ((T0 >> 1) + k + 1) << 1);
      unit = lo + (start >> 1), t0 = start & 1, tn = end - start;
    }
    Piece pc;
    pc.seg = unit / per_seg();
    const int r = unit - pc.seg * per_seg();
    pc.s = r / upg();
    const int q = r - pc.s * upg();  // 2 * group + half
    pc.grp = q >> 1;
    pc.t0 = 2 * (q & 1) + t0, pc.tn = tn;
    return pc;
  }
};

template <int kEpi>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ Job p, const __grid_constant__ WeightMaps maps) {
  static_assert(kEpi == kEpiGated || kEpi == kEpiRows, "grouped products only");
  constexpr int NT = 4;       // four 8-slot MMA columns: a segment's 32 slots
  constexpr int NI = 4;       // floats per accumulator column
  constexpr int V = NT * NI;  // accumulator floats per lane and tile
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;

  // ---- shared memory: warp w's stages at smem + w*ns*2304, one mbarrier per
  // stage, the staged rows (16 + the zero row), then the tables
  const int ns = p.ns;
  const size_t ring_bytes = static_cast<size_t>(kWarps) * ns * kStageBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + ring_bytes) + warp * ns;
  uint8_t* xs = smem + ring_bytes + static_cast<size_t>(kWarps) * ns * 8;
  const size_t xs_bytes = static_cast<size_t>(kPrefillSlots + 1) * (static_cast<size_t>(p.xs_chunks) * kXChunkBytes + 16);
  int* row_src = reinterpret_cast<int*>(xs + xs_bytes);  // [32] source row of each staged row
  int* sigma = row_src + kPrefillSlots;                   // [33] power-of-two scale of each staged row
  int* slot_row = sigma + kPrefillSlots + 1;              // [32] staged row of each slot
  int* slot_out = slot_row + kPrefillSlots;               // [32] output row of each slot, -1: none
  float* mul = reinterpret_cast<float*>(slot_out + kPrefillSlots);  // [32] global scale of the segment
  int* cur = reinterpret_cast<int*>(mul + kPrefillSlots) + warp * 8;  // this warp's copy cursor
  int* seg_list = reinterpret_cast<int*>(mul + kPrefillSlots) + kWarps * 8;  // [max_segs + 1] matrix
  int* seg_blk = seg_list + p.max_segs + 1;  // [max_segs + 1] block: pairs 32b .. 32b+31 of the matrix
  int* misc = seg_blk + p.max_segs + 1;      // [0] segments, [1] staged rows
  if ((smem_addr(smem) & 127u) || smem_addr(misc + 4) - smem_addr(smem) > dynamic_smem_bytes()) {
    // the carve-up does not fit the launch's shared memory (a plan error): touch nothing
    if (threadIdx.x == 0) atomicOr(&g_device_error, kErrPlan);
    return;
  }

  if (lane == 0) {
    for (int s = 0; s < ns; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // ---- segments: each expert's blocks of at most 32 pairs, then the shared
  // expert's blocks of at most 32 tokens
  if (!p.routing_ready) pdl_wait();
  if (warp == 0) {
    int n = 0;
    for (int base = 0; base < p.n_experts; base += 32) {
      const int e = base + lane;
      const int cnt = e < p.n_experts ? __ldg(p.offsets + e + 1) - __ldg(p.offsets + e) : 0;
      const int nb = (cnt + kPrefillSlots - 1) / kPrefillSlots;
      int incl = nb;  // inclusive prefix of the block counts over the warp
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      for (int b = 0, i = n + incl - nb; b < nb; ++b, ++i)
        if (i < p.max_segs) seg_list[i] = e, seg_blk[i] = b;
      n += __shfl_sync(0xffffffffu, incl, 31);
    }
    const int nsh = p.has_shared ? (p.m + kPrefillSlots - 1) / kPrefillSlots : 0;
    for (int b = lane; b < nsh; b += 32)
      if (n + b < p.max_segs) seg_list[n + b] = kSharedSeg, seg_blk[n + b] = b;
    n += nsh;
    if (lane == 0) {
      if (n > p.max_segs) atomicOr(&g_device_error, kErrPlan);  // the routing breaks its bounds
      misc[0] = min(n, p.max_segs);
    }
  }
  __syncthreads();
  const PrefillDeal pd{misc[0], p.S, p.L, p.kc, p.ng, static_cast<int>(gridDim.x)};
  int u0, u1;
  pd.cta_range(blockIdx.x, u0, u1);
  // run r: the CTA's units of (segment, slice) block b0 + r; its activation rows
  // are the segment's, over the slice's columns
  auto run_lo = [&](int r) { return pd.run_lo(u0, r); };
  auto run_hi = [&](int r) { return pd.run_hi(u0, u1, r); };
  auto run_seg = [&](int r) { return pd.run_seg(u0, r); };
  auto run_slice = [&](int r) { return pd.run_slice(u0, r); };
  const bool fits = p.L <= p.xs_chunks;
  if (!fits && threadIdx.x == 0) atomicOr(&g_device_error, kErrPlan);  // the plan does not cover a slice
  const int n_runs = fits ? pd.n_runs(u0, u1) : 0;

  // ---- warp w's pieces of run r (PrefillDeal::piece)
  struct Deal {
    int lo, nu, np;
  };
  auto deal_of = [&](int r) -> Deal {
    Deal d;
    d.lo = run_lo(r);
    d.nu = run_hi(r) - d.lo;
    d.np = pd.n_pieces(d.nu, warp);
    return d;
  };
  auto piece_at = [&](const Deal& d, int k) -> Piece { return pd.piece(d.lo, d.nu, warp, k); };
  auto slice_len = [&](int s) { return pd.slice_len(s); };

  // ---- producer (lane 0): cursor over this warp's pieces, run after run, ahead
  // of the consumer by the ring's depth.  A piece of tn tiles is TMA boxes of tn
  // tiles x copy_chunks(tn) chunks (2,304 bytes each).  Cursor (lane 0's, in
  // shared memory): [0] map index (tn-1, +4 for the shared expert), [1] first
  // tile, [2] next chunk, [3] group, [4] chunks per copy, [5] run, [6] next piece.
  int prem = 0;  // copies left in the open piece
  const uint64_t policy = l2_evict_first_policy();
  uint8_t* ring = smem + static_cast<size_t>(warp) * ns * kStageBytes;
  const uint32_t ring_s = smem_addr(ring), bar_s = smem_addr(bar);
  if (lane == 0) cur[5] = 0, cur[6] = 0;
  auto issue_next = [&](int stage) {
    if (prem == 0) {
      if (cur[5] >= n_runs) return;
      Deal d = deal_of(cur[5]);
      while (cur[6] >= d.np) {
        if (++cur[5] >= n_runs) return;
        d = deal_of(cur[5]);
        cur[6] = 0;
      }
      const Piece pc = piece_at(d, cur[6]++);
      const int e = seg_list[pc.seg];
      const int step = copy_chunks(pc.tn);
      prem = (slice_len(pc.s) + step - 1) / step;
      cur[0] = (pc.tn - 1) + (e == kSharedSeg ? 4 : 0);
      cur[1] = pc.t0;
      cur[2] = pc.s * p.L;
      cur[3] = (e >= 0 ? e * p.ng : 0) + pc.grp;  // group within the stack
      cur[4] = step;
    }
    const int mi = cur[0];
    const uint32_t b = bar_s + stage * 8;
    mbar_arrive_expect_tx_s(b, static_cast<uint32_t>(((mi & 3) + 1) * cur[4]) * kTileBytes);
    tma_load_4d_s(ring_s + stage * kStageBytes, mi < 4 ? &maps.w[mi] : &maps.sh[mi - 4], 0, cur[1], cur[2], cur[3], b,
                  policy);
    cur[2] += cur[4];
    --prem;
  };
  if (lane == 0)
    for (int st = 0; st < min(ns, p.npre); ++st) issue_next(st);

  // ---- run r's tables (thread j < 32: slot j of the segment): the source row
  // it stages (gate+up: the pair's token row of x; down: the pair's gate+up
  // output row), its output row, and the segment's global scale.  Empty slots
  // read the zero row (index = valid slots) and write nothing.  The down
  // product's routing is complete before its grid starts, so it builds run 0's
  // tables before the wait.
  auto build_tables = [&](int r) {
    if (threadIdx.x < kPrefillSlots && n_runs > 0) {
      const int j = threadIdx.x;
      const int e = seg_list[run_seg(r)], b = seg_blk[run_seg(r)];
      const int cnt = e == kSharedSeg ? p.m : __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
      const int v = min(kPrefillSlots, cnt - kPrefillSlots * b);  // valid slots (>= 1)
      int out = -1;
      if (j < v) {
        if (e == kSharedSeg) {
          out = p.m * p.top_k + kPrefillSlots * b + j;
          row_src[j] = p.x_by_pair ? out : kPrefillSlots * b + j;
        } else {
          out = __ldg(p.pairs + __ldg(p.offsets + e) + kPrefillSlots * b + j);
          row_src[j] = p.x_by_pair ? out : out / p.top_k;
        }
      }
      slot_row[j] = j < v ? j : v;
      slot_out[j] = out;
      mul[j] = e == kSharedSeg ? __ldg(p.gs_sh) : __ldg(p.gs + e);
      if (j == 0) misc[1] = v;
    }
  };
  int c_lo = 0, stride = 16, nrows = 0;
  // after build_tables(r) and a barrier: stage run r's rows over its slice's
  // columns (ends with a barrier)
  // the ring's stages past the first npre go out once the first run's activation
  // loads are issued (see the decode kernel)
  bool rest_issued = false;
  auto issue_rest = [&]() {
    if (!rest_issued) {
      rest_issued = true;
      if (lane == 0)
        for (int st = min(ns, p.npre); st < ns; ++st) issue_next(st);
    }
  };
  auto stage_run = [&](int r) {
    const int nch = n_runs > 0 ? slice_len(run_slice(r)) : 0;
    c_lo = n_runs > 0 ? run_slice(r) * p.L : 0;
    stride = nch * kXChunkBytes + 16;
    nrows = n_runs > 0 ? misc[1] : 0;
    stage_rows<true>(p.x, p.k, c_lo * kTileK, nch, nrows, row_src, sigma, xs, stride, issue_rest);
  };
  if (p.routing_ready) {
    build_tables(0);
    pdl_wait();
  }
  pdl_launch_dependents();
  if (!p.routing_ready) build_tables(0);
  __syncthreads();
  stage_run(0);

  const uint32_t xs_addr = smem_addr(xs);
  float acc[2][NT][NI];

  // Finish tile t (0..3) of group grp from a[] (output units).  MMA fragment:
  // column c holds slots c*8 + 2*t4 + (i & 1) of rows g (i < 2) and g + 8.
  auto finish_tile = [&](int grp, int t, const float (&a)[NT][NI]) {
    const int rb = grp * 4 + t;  // 16-row block within the matrix
#pragma unroll
    for (int c = 0; c < NT; ++c)
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int slot = c * 8 + 2 * t4 + (i & 1);
        const int out = slot_out[slot];
        if constexpr (kEpi == kEpiRows) {
          const int row = rb * 16 + g + 8 * (i >> 1);
          if (out >= 0 && row < p.n) p.yf[static_cast<size_t>(out) * p.yf_ld + row] = a[c][i];
        } else if (i < 2 && out >= 0) {  // gated: rows g = gate j, g + 8 = up j of block rb, j = rb*8 + g
          p.y[static_cast<size_t>(out) * p.y_ld + rb * 8 + g] = f32_to_bf16_bits(gelu_tanh(a[c][i]) * a[c][i + 2]);
        }
      }
  };

  const uint32_t ring_addr = smem_addr(ring);
  int st = 0;           // ring stage of the next copy
  uint32_t ph = 0;      // its mbarrier parity
  bool failed = false;  // a copy did not complete in time
  for (int r = 0; r < n_runs; ++r) {
    if (r > 0) {
      // the next run's rows replace the staged ones once every warp is done
      __syncthreads();
      build_tables(r);
      __syncthreads();
      stage_run(r);
    }
    const Deal d = deal_of(r);
    for (int k = 0; k < d.np && !failed; ++k) {
      const Piece pc = piece_at(d, k);
      const int nch = slice_len(pc.s);
      uint32_t xr[NT];
#pragma unroll
      for (int c = 0; c < NT; ++c) xr[c] = xs_addr + slot_row[c * 8 + g] * stride + t4 * 32;
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int c = 0; c < NT; ++c)
#pragma unroll
          for (int i = 0; i < NI; ++i) acc[a][c][i] = 0.f;
      // the piece's copies: copy j holds chunks j*step .. of the slice, TN tiles
      // each at stage + cc*TN*576
      auto stream_piece = [&](auto tn_c) {
        constexpr int TN = decltype(tn_c)::value;
        constexpr int kStep = copy_chunks(TN);
        for (int ch = 0; ch < nch; ch += kStep) {
          if (!mbar_wait_warp(&bar[st], ph)) {
            failed = true;
            return;
          }
          const uint32_t stage = ring_addr + st * kStageBytes;
          const int cnt = min(kStep, nch - ch);  // chunks of this copy inside the slice
          for (int cc = 0; cc < cnt; ++cc) {
            mma_chunk<NT, TN>(stage + cc * TN * kTileBytes, xr, lane, acc);
#pragma unroll
            for (int c = 0; c < NT; ++c) xr[c] += kXChunkBytes;
          }
          __syncwarp();
          if (lane == 0) {
            fence_proxy_async_smem();  // this warp's reads of the stage before the next copy into it
            issue_next(st);
          }
          if (++st == ns) st = 0, ph ^= 1u;
        }
      };
      if (pc.tn == 2)
        stream_piece(std::integral_constant<int, 2>{});
      else
        stream_piece(std::integral_constant<int, 1>{});
      if (failed) break;
      // ---- to output units: times g * 2^(8 - sigma of the slot's staged row)
      float mulv[NT][2];
#pragma unroll
      for (int c = 0; c < NT; ++c)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int slot = c * 8 + 2 * t4 + h;
          const int row = slot_row[slot];
          mulv[c][h] = row < nrows ? mul[slot] * exp2i(8 - sigma[row]) : 0.f;
        }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int c = 0; c < NT; ++c)
#pragma unroll
          for (int i = 0; i < NI; ++i) acc[a][c][i] *= mulv[c][i & 1];
      if (p.S == 1) {
#pragma unroll
        for (int a = 0; a < 2; ++a)
          if (a < pc.tn) finish_tile(pc.grp, pc.t0 + a, acc[a]);
      } else {
        // ---- k-split: per tile, store the partial and take a ticket; the last of
        // the S slices sums all S partials in slice order and finishes the tile
        const size_t cell0 = (static_cast<size_t>(pc.seg) * p.ng + pc.grp) * 4 + pc.t0;
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          if (a >= pc.tn) break;
          float* dst = p.fix + (((cell0 + a) * p.S + pc.s) * 32 + lane) * V;
#pragma unroll
          for (int c = 0; c < NT; ++c)
            __stcg(reinterpret_cast<float4*>(dst + c * 4), make_float4(acc[a][c][0], acc[a][c][1], acc[a][c][2], acc[a][c][3]));
        }
        __threadfence();
        __syncwarp();
        unsigned last = 0;  // bit a: this warp completed tile t0 + a
        if (lane == 0) {
#pragma unroll
          for (int a = 0; a < 2; ++a)
            if (a < pc.tn && atomicAdd(&p.fix_cnt[cell0 + a], 1u) == static_cast<unsigned>(p.S - 1)) {
              last |= 1u << a;
              atomicExch(&p.fix_cnt[cell0 + a], 0u);
            }
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) __threadfence();
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          if (!((last >> a) & 1u)) continue;
          float sum[NT][NI];
#pragma unroll
          for (int c = 0; c < NT; ++c)
#pragma unroll
            for (int i = 0; i < NI; ++i) sum[c][i] = 0.f;
          const float* src0 = p.fix + ((cell0 + a) * p.S * 32 + lane) * V;
          for (int s = 0; s < p.S; ++s) {
#pragma unroll
            for (int c = 0; c < NT; ++c) {
              const float4 f = __ldcg(reinterpret_cast<const float4*>(src0 + static_cast<size_t>(s) * 32 * V + c * 4));
              sum[c][0] += f.x, sum[c][1] += f.y, sum[c][2] += f.z, sum[c][3] += f.w;
            }
          }
          finish_tile(pc.grp, pc.t0 + a, sum);
        }
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

}  // namespace nvfp4
