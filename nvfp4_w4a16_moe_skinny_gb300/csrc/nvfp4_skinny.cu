// C-ABI entry points of the NVFP4 W4A16 skinny library (sm_103a).
// Host-side argument checks, launch geometry and kernel dispatch.  The kernels
// live in the included headers; everything is one translation unit.
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <cstdint>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "nvfp4_skinny.h"
#include "common.cuh"
#include "quant.cuh"
#include "launch.cuh"
#include "prefill.cuh"
#include "moe.cuh"

namespace nvfp4 {

namespace {

constexpr size_t kCounterBytes = 4096;   // arrival counters at the start of a workspace
constexpr int kMaxDevices = 64;

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cache[kMaxDevices] = {0};
  if (dev >= 0 && dev < kMaxDevices && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) cache[dev] = n;
  return n;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }


int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

nvfp4_status check_weight(const nvfp4_weight* w, int num_matrices, uint32_t flags) {
  if (!w || !w->data || !w->global_scale) return NVFP4_ERR_NULL;
  if (w->layout_version != NVFP4_LAYOUT_VERSION || w->flags != flags) return NVFP4_ERR_LAYOUT;
  if (w->n < 1 || w->k < 16 || (w->k % 16) || w->num_matrices != num_matrices) return NVFP4_ERR_SHAPE;
  if (!aligned(w->data, 16) || !aligned(w->global_scale, 4)) return NVFP4_ERR_ALIGN;
  return NVFP4_OK;
}

// ------------------------------------------------------------------ streaming-kernel plans
// The K split S is chosen from the shapes alone, against a fixed reference
// parallelism (152 SMs x 16 warps), so workspace sizes are host-computable and
// identical on every device; the grid is the device's SM count, and the staging
// capacities are sized for that grid.
constexpr int kPlanSMs = 152;
constexpr int kMaxSplit = 16;


bool use_mma(int m) { return m >= 2; }  // (the decode kernel's instance for m; see dispatch_stream)
// accumulator floats per lane and 16-row tile (the fixup partial of one tile)
int acc_per_tile(int m) { return use_mma(m) ? (m <= 8 ? 4 : 8) : 2 * m; }

// A fixup area is a fixed 512 KiB of arrival counters (one per segment x group x
// tile, at most 131,072) followed by the partials.  The counters sit at the same
// place whatever the shape, and every call leaves them zero, so one zero-filled
// workspace can serve calls of different shapes.
constexpr size_t kFixCounterBytes = 512 * 1024;

// Partial floats per lane and tile: the decode kernel's accumulator, or the
// prefill kernel's four 8-slot MMA columns (m > 16).
size_t fixup_bytes(int m, int S, int ng, int n_seg_max) {
  if (S <= 1) return 0;
  return kFixCounterBytes +
         static_cast<size_t>(n_seg_max) * ng * 4 * S * 32 * (m > 16 ? 16 : acc_per_tile(m)) * sizeof(float);
}

// Launch plan for split S on a grid of multiples of `sms` CTAs: one CTA per SM
// (more, in waves, if a CTA would otherwise stage the rows of more than
// kMaxCtaSegs segments, or more rows than fit beside a ring -- only on devices
// with few SMs), staging capacities that cover the busiest CTA, then the deepest
// ring that fits in shared memory.
// n_seg_max is the most segments the job can have (the capacity of the
// segment list); n_experts sizes the decode kernel's expert table; per_run: the
// prefill kernel, which stages one segment's 16 rows at a time.
bool make_plan(int m, int S, int ng, int kc, int n_seg_max, int n_experts, bool per_run, bool x_by_pair, int sms,
               Plan* out) {
  const int L = ceil_div(kc, S);
  if (per_run) {
    // the prefill kernel: a run never crosses a slice, so the staged rows (32 and
    // the zero row) cover one slice; one CTA per SM
    for (int ns = 8; ns >= 2; --ns) {
      const size_t smem = prefill_smem_bytes(L, ns, n_seg_max);
      if (smem <= kMaxSmem) {
        *out = Plan{S, L, ns, L, kPrefillSlots, 1, sms, n_seg_max, true, smem};
        return true;
      }
    }
    return false;
  }
  const int per_seg = S * ng;
  // a single matrix split along K on a grid that S divides: every CTA stays inside
  // one slice (DecodeDeal::cta_range) and stages that slice's columns only
  const bool slice_ctas = n_seg_max == 1 && !x_by_pair && S > 1 && sms % S == 0;
  int prev_segs = -1;
  for (int grid = sms;; grid += sms) {
    const long long nu_max = (static_cast<long long>(n_seg_max) * per_seg + grid - 1) / grid;
    const int segs = static_cast<int>(std::min<long long>(n_seg_max, (nu_max + per_seg - 1) / per_seg + 1));
    if (segs > kMaxCtaSegs) continue;
    int xs_chunks = kc;
    if (slice_ctas && grid == sms) {
      xs_chunks = L;
    } else if (segs == 1) {
      const long long nu_seg = std::min<long long>(nu_max, per_seg);  // units of one run
      xs_chunks = static_cast<int>(std::min<long long>(kc, ((nu_seg + ng - 1) / ng + 1) * L));
    }
    const int xs_rows = x_by_pair ? segs * std::min(m, 16) : m;
    for (int ns = 8; ns >= 2; --ns) {
      const size_t smem = stream_smem_bytes(xs_rows, xs_chunks, ns, n_experts);
      if (smem <= kMaxSmem) {
        *out = Plan{S, L, ns, xs_chunks, xs_rows, std::min(segs, kMaxCtaSegs), grid, n_seg_max, per_run, smem,
                    slice_ctas && grid == sms};
        return true;
      }
    }
    // staging the rows of fewer segments per CTA (a larger grid) is the only
    // way left to fit; stop once the grid no longer lowers the count
    if (!x_by_pair || segs == prev_segs) return false;
    prev_segs = segs;
  }
}

// Predicted time (us) of one launch of `plan` over n_seg segments of ng groups,
// on the reference grid, for ranking the splits: a fixed launch cost, staging
// the activations over the columns a CTA touches, the busiest warp's
// tile-chunks (whole units amortise the x loads over four tiles and run
// faster per tile than split tiles) or the SM's share of HBM, whichever is
// slower, and, when K is split, a fence + ticket per piece and the last
// slice's reads of the S partials a few at a time.  The constants are fitted to
// measured launches of the dense and MoE products on GB300.
double plan_cost(int m_tokens, int ng, int n_seg, bool x_by_pair, const Plan& plan) {
  const int m = std::min(m_tokens, 16);  // token slots of one segment
  const int S = plan.S, L = plan.L;
  const long long units = static_cast<long long>(n_seg) * S * ng;
  const long long nu = (units + kPlanSMs - 1) / kPlanSMs;  // units of the busiest CTA
  const bool mma = use_mma(m);
  // the busiest warp: its whole units (round-robin) and its share of the rest's tiles
  const int nw = whole_units(static_cast<int>(nu));
  const long long whole = (nw + kWarps - 1) / kWarps;
  const long long split_tiles = (kChunkTiles * (nu - nw) + kWarps - 1) / kWarps;
  const long long pieces = whole + std::min<long long>(2, split_tiles);
  const double per_whole = mma ? 0.26 : 0.22, per_split = mma ? 0.30 : 0.25;  // us per tile-chunk
  const double tc_time = (whole * kChunkTiles * per_whole + split_tiles * per_split) * L;
  const int rows = plan.per_run ? 16 : (x_by_pair ? m * std::min(plan.max_cta_segs, 2) : m);
  const double span = plan.slice_ctas ? L : std::min<double>(plan.xs_chunks, L * (1.0 + static_cast<double>(nu - 1) / ng));
  const double t_stage = 1.0 + rows * span * kXChunkBytes / 30000.0;
  const double t_warp = tc_time;
  const double t_mem = static_cast<double>(nu) * L * kStageBytes / 40000.0;  // 40 GB/s per SM
  const int v = acc_per_tile(m), batch = v >= 12 ? 1 : (v >= 8 ? 2 : 4);
  const double t_fix = S > 1 ? 1.5 * pieces + 1.5 * ((S + batch - 1) / batch) : 0.0;
  return 3.0 + t_stage + std::max(t_warp, t_mem) + t_fix;
}

// S for a job: the cheapest by plan_cost (ties to the smaller S), planned on the
// reference grid so that it depends on the shapes only.  n_seg_est is the
// expected number of segments, n_seg_max the most there can be.
int choose_split_uncached(int m, int ng, int kc, int n_seg_est, int n_seg_max, int n_experts, bool per_run,
                          bool x_by_pair, bool allow_split) {
  int best = 1;
  double best_cost = 1e30;
  Plan pl;
  if (per_run) {
    // the prefill kernel: the smallest split whose slice of 32 staged rows fits
    // (each further split only adds fixup traffic)
    for (int s = 1; s <= std::min(kMaxSplit, kc); ++s) {
      if (s > 1 && (!allow_split || static_cast<size_t>(n_seg_max) * ng * 4 > kFixCounterBytes / sizeof(unsigned)))
        break;
      if (make_plan(m, s, ng, kc, n_seg_max, n_experts, true, x_by_pair, kPlanSMs, &pl)) return s;
    }
    return 1;
  }
  if (make_plan(m, 1, ng, kc, n_seg_max, n_experts, per_run, x_by_pair, kPlanSMs, &pl))
    best_cost = plan_cost(m, ng, n_seg_est, x_by_pair, pl);
  if (!allow_split) return 1;
  if (static_cast<size_t>(n_seg_max) * ng * 4 > kFixCounterBytes / sizeof(unsigned)) return 1;
  for (int s = 2; s <= std::min(kMaxSplit, kc); ++s) {
    const int L = ceil_div(kc, s);
    if (ceil_div(kc, L) != s) continue;  // the same slices as a smaller S
    if (!make_plan(m, s, ng, kc, n_seg_max, n_experts, per_run, x_by_pair, kPlanSMs, &pl)) continue;
    const double c = plan_cost(m, ng, n_seg_est, x_by_pair, pl);
    if (c < best_cost * 0.99) best = s, best_cost = c;
  }
  return best;
}

// choose_split, remembered per argument set (it depends on the shapes only).
int choose_split(int m, int ng, int kc, int n_seg_est, int n_seg_max, int n_experts, bool per_run, bool x_by_pair,
                 bool allow_split) {
  static std::mutex mu;
  static std::map<std::array<int, 9>, int> memo;
  const std::array<int, 9> key{m,         ng, kc, n_seg_est, n_seg_max, n_experts, per_run ? 1 : 0, x_by_pair ? 1 : 0,
                               allow_split ? 1 : 0};
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = memo.find(key);
    if (it != memo.end()) return it->second;
  }
  const int s = choose_split_uncached(m, ng, kc, n_seg_est, n_seg_max, n_experts, per_run, x_by_pair, allow_split);
  std::lock_guard<std::mutex> lock(mu);
  if (memo.size() > 4096) memo.clear();
  memo[key] = s;
  return s;
}

// ------------------------------------------------------------------ TMA tensor maps
// cuTensorMapEncodeTiled is a driver-API function; the library reaches it through
// the runtime's entry-point query, so it links only the runtime.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// The four tensor maps (boxes of 1..4 tiles, see WeightMaps) of the repacked
// weight stack `w`: num_matrices x ceil(n/64) groups of ceil(k/64) chunks.
bool encode_weight_maps(const nvfp4_weight* w, CUtensorMap (&maps)[4]) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const int kc = ceil_div(w->k, kTileK);
  const cuuint64_t groups = static_cast<cuuint64_t>(w->num_matrices) * ceil_div(w->n, kGroupRows);
  const cuuint64_t dims[4] = {kTileBytes / 8, kChunkTiles, static_cast<cuuint64_t>(kc), groups};
  const cuuint64_t strides[3] = {kTileBytes, kStageBytes, static_cast<cuuint64_t>(kc) * kStageBytes};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  for (int tn = 1; tn <= 4; ++tn) {
    const cuuint32_t box[4] = {kTileBytes / 8, static_cast<cuuint32_t>(tn), static_cast<cuuint32_t>(copy_chunks(tn)), 1};
    if (fn(&maps[tn - 1], CU_TENSOR_MAP_DATA_TYPE_UINT64, 4, const_cast<void*>(w->data), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

// The maps of one weight, remembered per (device, address, shape): a weight is
// repacked once and used for many calls.  The cache holds encodings only (no
// device memory); at most 1024 entries, then it starts over.
bool weight_maps_cached(const nvfp4_weight* w, CUtensorMap (&maps)[4]) {
  struct Entry {
    CUtensorMap m[4];
  };
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int, int, int>, Entry> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const auto key = std::make_tuple(dev, w->data, w->n, w->k, w->num_matrices);
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) {
      for (int i = 0; i < 4; ++i) maps[i] = it->second.m[i];
      return true;
    }
  }
  if (!encode_weight_maps(w, maps)) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() >= 1024) cache.clear();
  Entry& e = cache[key];
  for (int i = 0; i < 4; ++i) e.m[i] = maps[i];
  return true;
}

// Maps of a weight and, for a MoE layer, of its shared expert.
bool make_maps(const nvfp4_weight* w, const nvfp4_weight* shared, WeightMaps* out) {
  if (!weight_maps_cached(w, out->w)) return false;
  if (shared) return weight_maps_cached(shared, out->sh);
  for (int i = 0; i < 4; ++i) out->sh[i] = out->w[i];
  return true;
}

void set_fixup(Job* p, void* base) {
  p->fix_cnt = static_cast<unsigned*>(base);
  p->fix = reinterpret_cast<float*>(static_cast<uint8_t*>(base) + kFixCounterBytes);
}

Job dense_job(const nvfp4_weight* w, const uint16_t* x, int m) {
  Job p{};
  p.w = static_cast<const uint8_t*>(w->data);
  p.gs = w->global_scale;
  p.n = w->n, p.k = w->k;
  p.ng = ceil_div(w->n, kGroupRows), p.kc = ceil_div(w->k, kTileK);
  p.x = x;
  p.m = m;
  return p;
}

int dense_split(int m, int n, int k) {
  return choose_split(m, ceil_div(n, kGroupRows), ceil_div(k, kTileK), 1, 1, 0, false, false, true);
}

// The failure path of the bounded waits, without a fault: every warp of one CTA
// waits, with the kernels' warp-collective wait, on an mbarrier phase that no
// thread completes (no copy is attached to it), gives up after `limit` cycles,
// records kErrWaitTimeout and returns.
__global__ void __launch_bounds__(128) selftest_wait_kernel(long long limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  (void)mbar_wait_warp(&bar, 0, limit);
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

const char* nvfp4_status_string(nvfp4_status st) {
  switch (st) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_NULL: return "null pointer";
    case NVFP4_ERR_SHAPE: return "bad shape";
    case NVFP4_ERR_ALIGN: return "misaligned pointer";
    case NVFP4_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4_ERR_LAYOUT: return "weight layout version or flags mismatch";
    case NVFP4_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

uint32_t nvfp4_layout_version(void) { return NVFP4_LAYOUT_VERSION; }

nvfp4_status nvfp4_selftest_wait_timeout(int64_t limit_cycles, cudaStream_t stream) {
  if (limit_cycles < 1 || limit_cycles > (int64_t{1} << 31)) return NVFP4_ERR_SHAPE;
  selftest_wait_kernel<<<1, 128, 0, stream>>>(static_cast<long long>(limit_cycles));
  return launched();
}

nvfp4_status nvfp4_device_error(uint32_t* out, int32_t clear) {
  if (!out) return NVFP4_ERR_NULL;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (clear) {
    const unsigned z = 0;
    if (cudaMemcpyToSymbol(g_device_error, &z, sizeof(z)) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  // the streaming kernels' translation units, one per epilogue
  for (auto fn : {epi_error_word<kEpiStore>, epi_error_word<kEpiArgmax>, epi_error_word<kEpiGated>,
                  epi_error_word<kEpiRows>, epi_error_word<kEpiSample>}) {
    uint32_t w = 0;
    if (const nvfp4_status st = fn(&w, clear)) return st;
    v |= w;
  }
  *out = v;
  return NVFP4_OK;
}

size_t nvfp4_repacked_bytes(int32_t n, int32_t k, int32_t num_matrices) {
  if (n < 1 || k < 16 || (k % 16) || num_matrices < 1) return 0;
  const size_t nb = static_cast<size_t>(ceil_div(n, kGroupRows)) * (kGroupRows / kTileRows);
  const size_t kc = static_cast<size_t>(ceil_div(k, kTileK));
  return static_cast<size_t>(num_matrices) * nb * kc * kTileBytes;
}

size_t nvfp4_quantize_workspace_bytes(int32_t num_matrices) {
  return num_matrices < 1 ? 0 : static_cast<size_t>(num_matrices) * sizeof(unsigned);
}

}  // extern "C"

namespace nvfp4 {
namespace {

// The quantizer's two grids over num_matrices matrices of [n, k] elements of T
// (fp32 weights or bf16 activation rows): per-matrix amax, then the codes.
template <typename T>
nvfp4_status quantize_launch(const T* w, int32_t num_matrices, int32_t n, int32_t k, uint8_t* nibbles,
                             uint8_t* scales, float* global_scale, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!w || !nibbles || !scales || !global_scale) return NVFP4_ERR_NULL;
  if (num_matrices < 1 || n < 1 || k < 16 || (k % 16)) return NVFP4_ERR_SHAPE;
  if (!ws || ws_bytes < nvfp4_quantize_workspace_bytes(num_matrices)) return NVFP4_ERR_WORKSPACE;
  if (!aligned(w, 16) || !aligned(nibbles, 8) || !aligned(global_scale, 4) || !aligned(ws, 4)) return NVFP4_ERR_ALIGN;
  unsigned* amax = static_cast<unsigned*>(ws);
  if (cudaMemsetAsync(amax, 0, sizeof(unsigned) * num_matrices, stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  const size_t per = static_cast<size_t>(n) * k;
  const int sms = std::max(1, sm_count());
  const int bx = static_cast<int>(std::min<size_t>((per + 255) / 256, static_cast<size_t>(sms) * 4));
  quant_amax_kernel<T><<<dim3(bx, num_matrices), 256, 0, stream>>>(w, per, amax);
  if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  const size_t groups = per / 16;
  const int gx = static_cast<int>(std::min<size_t>((groups + 255) / 256, static_cast<size_t>(sms) * 8));
  quant_groups_kernel<T><<<dim3(gx, num_matrices), 256, 0, stream>>>(w, n, k, amax, nibbles, scales, global_scale);
  return launched();
}

}  // namespace
}  // namespace nvfp4

extern "C" {

nvfp4_status nvfp4_quantize(const float* w, int32_t num_matrices, int32_t n, int32_t k, uint8_t* nibbles,
                            uint8_t* scales, float* global_scale, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return quantize_launch(w, num_matrices, n, k, nibbles, scales, global_scale, ws, ws_bytes, stream);
}

nvfp4_status nvfp4_quantize_act(const uint16_t* x, int32_t m, int32_t k, uint8_t* codes, uint8_t* scales,
                                float* global_scale, void* ws, size_t ws_bytes, cudaStream_t stream) {
  // each token row is a matrix of its own (one global scale per row): one grid,
  // one CTA per row; the workspace is not needed but checked as for nvfp4_quantize
  if (!x || !codes || !scales || !global_scale) return NVFP4_ERR_NULL;
  if (m < 1 || m > 4096 || k < 16 || (k % 16)) return NVFP4_ERR_SHAPE;
  if (!ws || ws_bytes < nvfp4_quantize_workspace_bytes(m)) return NVFP4_ERR_WORKSPACE;
  if (!aligned(x, 16) || !aligned(codes, 8) || !aligned(global_scale, 4)) return NVFP4_ERR_ALIGN;
  if (launch_pdl(quant_act_rows_kernel, dim3(m), dim3(kActQuantThreads), 0, stream, x, static_cast<int>(k), codes,
                 scales, global_scale) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  return launched();
}

nvfp4_status nvfp4_repack(const uint8_t* nibbles, const uint8_t* scales, int32_t num_matrices, int32_t n, int32_t k,
                          uint32_t flags, void* out, cudaStream_t stream) {
  if (!nibbles || !scales || !out) return NVFP4_ERR_NULL;
  if (num_matrices < 1 || n < 1 || k < 16 || (k % 16)) return NVFP4_ERR_SHAPE;
  if (flags & ~NVFP4_GATED) return NVFP4_ERR_LAYOUT;
  const bool gated = flags & NVFP4_GATED;
  if (gated && (n % kGroupRows)) return NVFP4_ERR_SHAPE;
  if (!aligned(out, 16)) return NVFP4_ERR_ALIGN;
  const int ng = ceil_div(n, kGroupRows), kc = ceil_div(k, kTileK);
  const size_t tiles = static_cast<size_t>(num_matrices) * ng * kc * 4;
  const int sms = std::max(1, sm_count());
  const int gx = static_cast<int>(std::min<size_t>((tiles * 36 + 255) / 256, static_cast<size_t>(sms) * 16));
  repack_kernel<<<gx, 256, 0, stream>>>(nibbles, scales, n, k, ng, kc, gated, tiles, static_cast<uint8_t*>(out));
  return launched();
}

nvfp4_status nvfp4_repack_host(const uint8_t* nibbles, const uint8_t* scales, int32_t num_matrices, int32_t n,
                               int32_t k, uint32_t flags, void* out, size_t out_bytes) {
  if (!nibbles || !scales || !out) return NVFP4_ERR_NULL;
  if (num_matrices < 1 || n < 1 || k < 16 || (k % 16)) return NVFP4_ERR_SHAPE;
  if (flags & ~NVFP4_GATED) return NVFP4_ERR_LAYOUT;
  const bool gated = flags & NVFP4_GATED;
  if (gated && (n % kGroupRows)) return NVFP4_ERR_SHAPE;
  if (out_bytes < nvfp4_repacked_bytes(n, k, num_matrices)) return NVFP4_ERR_WORKSPACE;
  const int ng = ceil_div(n, kGroupRows), kc = ceil_div(k, kTileK);
  const size_t chunks = static_cast<size_t>(num_matrices) * ng * kc * 4 * 36;
  uint8_t* dst = static_cast<uint8_t*>(out);
  for (size_t c = 0; c < chunks; ++c) {
    uint32_t words[4];
    repack_chunk(nibbles, scales, n, k, ng, kc, gated, c, words);
    for (int i = 0; i < 4; ++i)
      for (int b = 0; b < 4; ++b) dst[16 * c + 4 * i + b] = static_cast<uint8_t>(words[i] >> (8 * b));
  }
  return NVFP4_OK;
}

size_t nvfp4_gemm_workspace_bytes(int32_t m, int32_t n, int32_t k) {
  if (m < 1 || m > 16 || n < 1 || k < 16) return 0;
  return std::max<size_t>(16, fixup_bytes(m, dense_split(m, n, k), ceil_div(n, kGroupRows), 1));
}

nvfp4_status nvfp4_gemm(const nvfp4_weight* w, const uint16_t* x, int32_t m, uint16_t* y, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  if (const nvfp4_status st = check_weight(w, 1, 0)) return st;
  if (!x || !y) return NVFP4_ERR_NULL;
  if (m < 1 || m > 16) return NVFP4_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(y, 4)) return NVFP4_ERR_ALIGN;
  if (!ws || ws_bytes < nvfp4_gemm_workspace_bytes(m, w->n, w->k)) return NVFP4_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return NVFP4_ERR_ALIGN;
  Job p = dense_job(w, x, m);
  p.y = y;
  p.y_ld = w->n;
  set_fixup(&p, ws);
  Plan plan;
  if (!make_plan(m, dense_split(m, w->n, w->k), p.ng, p.kc, 1, 0, false, false, std::max(1, sm_count()), &plan))
    return NVFP4_ERR_SHAPE;
  WeightMaps maps;
  if (!make_maps(w, nullptr, &maps)) return NVFP4_ERR_CUDA;
  return dispatch_stream<kEpiStore>(p, maps, plan, stream);
}

nvfp4_status nvfp4_gemm_w4a4(const nvfp4_weight* w, const uint8_t* x_codes, const uint8_t* x_scales,
                             const float* x_global, int32_t m, uint16_t* y, void* ws, size_t ws_bytes,
                             cudaStream_t stream) {
  if (const nvfp4_status st = check_weight(w, 1, 0)) return st;
  if (!x_codes || !x_scales || !x_global || !y) return NVFP4_ERR_NULL;
  if (m < 1 || m > 16) return NVFP4_ERR_SHAPE;
  if (!aligned(x_codes, 16) || !aligned(x_global, 4) || !aligned(y, 4)) return NVFP4_ERR_ALIGN;
  if (!ws || ws_bytes < nvfp4_gemm_workspace_bytes(m, w->n, w->k)) return NVFP4_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return NVFP4_ERR_ALIGN;
  Job p = dense_job(w, nullptr, m);
  p.xq = x_codes, p.xq_sc = x_scales, p.xq_g = x_global;
  p.y = y;
  p.y_ld = w->n;
  set_fixup(&p, ws);
  Plan plan;
  if (!make_plan(m, dense_split(m, w->n, w->k), p.ng, p.kc, 1, 0, false, false, std::max(1, sm_count()), &plan))
    return NVFP4_ERR_SHAPE;
  WeightMaps maps;
  if (!make_maps(w, nullptr, &maps)) return NVFP4_ERR_CUDA;
  return dispatch_stream<kEpiStore>(p, maps, plan, stream);
}

nvfp4_status moe_router_logits(const nvfp4_weight* w, const uint16_t* x, int32_t m, const float* gate_scale, float eps,
                               float* logits, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (const nvfp4_status st = check_weight(w, 1, 0)) return st;
  if (!x || !logits) return NVFP4_ERR_NULL;
  if (m < 1 || m > 16 || w->n > 1024 || !(eps >= 0.f) || !(eps < INFINITY)) return NVFP4_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(logits, 4) || (gate_scale && !aligned(gate_scale, 4))) return NVFP4_ERR_ALIGN;
  if (!ws || ws_bytes < nvfp4_gemm_workspace_bytes(m, w->n, w->k)) return NVFP4_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return NVFP4_ERR_ALIGN;
  // the router matmul (the skinny GEMM with fp32 output), then the normalisation
  Job p = dense_job(w, x, m);
  p.yf = logits;
  p.yf_ld = w->n;
  set_fixup(&p, ws);
  Plan plan;
  if (!make_plan(m, dense_split(m, w->n, w->k), p.ng, p.kc, 1, 0, false, false, std::max(1, sm_count()), &plan))
    return NVFP4_ERR_SHAPE;
  WeightMaps maps;
  if (!make_maps(w, nullptr, &maps)) return NVFP4_ERR_CUDA;
  if (const nvfp4_status st = dispatch_stream<kEpiStore>(p, maps, plan, stream)) return st;
  constexpr int kWarpsPerCta = 4;
  if (launch_pdl(moe_router_norm_kernel, dim3(ceil_div(m, kWarpsPerCta)), dim3(32 * kWarpsPerCta), 0, stream, logits,
                 static_cast<int>(m), static_cast<int>(w->n), gate_scale, eps) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  return launched();
}

size_t lm_head_workspace_bytes(int32_t m, int32_t vocab) {
  if (m < 1 || m > 16 || vocab < 1) return 0;
  return kCounterBytes;  // the arrival counter and the per-token packed maxima
}

}  // extern "C"

namespace nvfp4 {
namespace {

// The lm_head never splits K: a split would put partial logits in memory.
// The lm_head grid: greedy argmax, or (temperature > 0) the Gumbel-max sample.
nvfp4_status lm_head_launch(const nvfp4_weight* w, const uint16_t* x, int32_t m, float* max_logit, int32_t* argmax,
                            void* ws, cudaStream_t stream, float temperature = 0.f, uint64_t seed = 0,
                            float softcap = 0.f, const uint8_t* xq = nullptr, const uint8_t* xq_sc = nullptr,
                            const float* xq_g = nullptr) {
  Job p = dense_job(w, x, m);
  p.xq = xq, p.xq_sc = xq_sc, p.xq_g = xq_g;
  p.softcap = softcap;
  p.am_cnt = static_cast<unsigned*>(ws);
  p.am_key = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(ws) + 64);
  p.max_logit = max_logit;
  p.argmax = argmax;
  Plan plan;
  if (!make_plan(m, 1, p.ng, p.kc, 1, 0, false, false, std::max(1, sm_count()), &plan)) return NVFP4_ERR_SHAPE;
  WeightMaps maps;
  if (!make_maps(w, nullptr, &maps)) return NVFP4_ERR_CUDA;
  if (temperature > 0.f) {
    p.inv_temp = 1.f / temperature;
    p.seed_lo = static_cast<uint32_t>(seed), p.seed_hi = static_cast<uint32_t>(seed >> 32);
    return dispatch_stream<kEpiSample>(p, maps, plan, stream);
  }
  return dispatch_stream<kEpiArgmax>(p, maps, plan, stream);
}

}  // namespace
}  // namespace nvfp4

extern "C" {

nvfp4_status lm_head_argmax(const nvfp4_weight* w, const uint16_t* x, int32_t m, float* max_logit, int32_t* argmax,
                            void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (const nvfp4_status st = check_weight(w, 1, 0)) return st;
  if (!x || !max_logit || !argmax) return NVFP4_ERR_NULL;
  if (m < 1 || m > 16) return NVFP4_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(max_logit, 4) || !aligned(argmax, 4)) return NVFP4_ERR_ALIGN;
  if (!ws || ws_bytes < lm_head_workspace_bytes(m, w->n)) return NVFP4_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return NVFP4_ERR_ALIGN;
  return lm_head_launch(w, x, m, max_logit, argmax, ws, stream);
}

nvfp4_status lm_head_argmax_w4a4(const nvfp4_weight* w, const uint8_t* x_codes, const uint8_t* x_scales,
                                 const float* x_global, int32_t m, float* max_logit, int32_t* argmax, void* ws,
                                 size_t ws_bytes, cudaStream_t stream) {
  if (const nvfp4_status st = check_weight(w, 1, 0)) return st;
  if (!x_codes || !x_scales || !x_global || !max_logit || !argmax) return NVFP4_ERR_NULL;
  if (m < 1 || m > 16) return NVFP4_ERR_SHAPE;
  if (!aligned(x_codes, 16) || !aligned(x_global, 4) || !aligned(max_logit, 4) || !aligned(argmax, 4))
    return NVFP4_ERR_ALIGN;
  if (!ws || ws_bytes < lm_head_workspace_bytes(m, w->n)) return NVFP4_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return NVFP4_ERR_ALIGN;
  return lm_head_launch(w, nullptr, m, max_logit, argmax, ws, stream, 0.f, 0, 0.f, x_codes, x_scales, x_global);
}

nvfp4_status lm_head_sample(const nvfp4_weight* w, const uint16_t* x, int32_t m, float temperature, uint64_t seed,
                            float* max_key, int32_t* token, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (const nvfp4_status st = check_weight(w, 1, 0)) return st;
  if (!x || !max_key || !token) return NVFP4_ERR_NULL;
  if (m < 1 || m > 16 || !(temperature >= 0.f) || !(temperature < INFINITY)) return NVFP4_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(max_key, 4) || !aligned(token, 4)) return NVFP4_ERR_ALIGN;
  if (!ws || ws_bytes < lm_head_workspace_bytes(m, w->n)) return NVFP4_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return NVFP4_ERR_ALIGN;
  return lm_head_launch(w, x, m, max_key, token, ws, stream, temperature, seed);
}

nvfp4_status lm_head_sample_ex(const nvfp4_weight* w, const uint16_t* x, int32_t m, float softcap, float temperature,
                               uint64_t seed, float* max_key, int32_t* token, void* ws, size_t ws_bytes,
                               cudaStream_t stream) {
  if (!(softcap >= 0.f) || !(softcap < INFINITY)) return NVFP4_ERR_SHAPE;
  if (const nvfp4_status st = check_weight(w, 1, 0)) return st;
  if (!x || !max_key || !token) return NVFP4_ERR_NULL;
  if (m < 1 || m > 16 || !(temperature >= 0.f) || !(temperature < INFINITY)) return NVFP4_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(max_key, 4) || !aligned(token, 4)) return NVFP4_ERR_ALIGN;
  if (!ws || ws_bytes < lm_head_workspace_bytes(m, w->n)) return NVFP4_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return NVFP4_ERR_ALIGN;
  return lm_head_launch(w, x, m, max_key, token, ws, stream, temperature, seed, softcap);
}

}  // extern "C"

// ------------------------------------------------------------------ MoE
namespace nvfp4 {
namespace {

size_t align16(size_t b) { return (b + 15) & ~static_cast<size_t>(15); }

// Segments of a MoE job: each expert that received pairs contributes one
// segment per block of its pairs -- one block when m <= 16 (the decode kernel),
// blocks of at most 32 otherwise (the prefill kernel) -- and the shared expert
// one per block of tokens of the same size.  expected_segments is the planning
// estimate under uniform routing (each expert's count binomial), and
// max_segments the most any routing can produce.
int segment_block(int m) { return m > 16 ? kPrefillSlots : 16; }

int expected_segments(int m, int top_k, int n_experts, bool shared) {
  const int blk = segment_block(m);
  const double q = static_cast<double>(top_k) / n_experts;
  double blocks = 0.0, pmf = std::pow(1.0 - q, m);  // P(count = 0)
  for (int c = 1; c <= m; ++c) {
    pmf *= (static_cast<double>(m - c + 1) / c) * (q / (1.0 - q));
    blocks += pmf * ((c + blk - 1) / blk);
    if (c > 64 && pmf < 1e-12) break;
  }
  const int est = static_cast<int>(n_experts * blocks + 0.5);
  return std::max(1, est) + (shared ? (m + blk - 1) / blk : 0);
}

int max_segments(int m, int top_k, int n_experts, bool shared) {
  const int blk = segment_block(m);
  const int pairs = m * top_k;
  const int experts = std::min(n_experts, pairs) + (m > 16 ? (pairs + blk - 1) / blk : 0);
  return experts + (shared ? (m + blk - 1) / blk : 0);
}

struct MoESplits {
  int s_gu, s_dn, n_seg_max;
  bool per_run;  // both products stage each segment's rows in turn (m > 16)
};

MoESplits moe_splits(int m, int top_k, int n_experts, int d, int inter, bool shared) {
  const int n_seg_est = expected_segments(m, top_k, n_experts, shared);
  MoESplits r;
  r.n_seg_max = max_segments(m, top_k, n_experts, shared);
  r.per_run = m > 16;
  r.s_gu = choose_split(m, ceil_div(2 * inter, kGroupRows), ceil_div(d, kTileK), n_seg_est, r.n_seg_max, n_experts,
                        r.per_run, false, true);
  r.s_dn = choose_split(m, ceil_div(d, kGroupRows), ceil_div(inter, kTileK), n_seg_est, r.n_seg_max, n_experts,
                        r.per_run, true, true);
  return r;
}

struct MoEWorkspace {
  size_t h, d, fix, total;
};

MoEWorkspace moe_workspace(int m, int top_k, int n_experts, int d, int inter, bool shared) {
  const MoESplits sp = moe_splits(m, top_k, n_experts, d, inter, shared);
  const size_t pairs = static_cast<size_t>(m) * top_k + m;
  MoEWorkspace w;
  w.h = align16(pairs * inter * sizeof(uint16_t));
  w.d = align16(pairs * d * sizeof(float));
  // gate_up and down share one fixup area (the down launch starts after gate_up
  // ends).  It comes first and always holds the arrival counters, so they sit at
  // the same offset whatever the shape: a zeroed workspace then serves calls of
  // any shape, each leaving the counters zero.
  w.fix = align16(std::max({kFixCounterBytes, fixup_bytes(m, sp.s_gu, ceil_div(2 * inter, kGroupRows), sp.n_seg_max),
                            fixup_bytes(m, sp.s_dn, ceil_div(d, kGroupRows), sp.n_seg_max)}));
  w.total = w.fix + w.h + w.d;
  return w;
}

}  // namespace
}  // namespace nvfp4

extern "C" {

nvfp4_status moe_route_topk(const float* logits, int32_t m, int32_t n_experts, int32_t top_k, int32_t* ids,
                            float* probs, int32_t* expert_offsets, int32_t* sorted_pairs, cudaStream_t stream) {
  return moe_route_topk_ex(logits, m, n_experts, top_k, 0, nullptr, ids, probs, expert_offsets, sorted_pairs, stream);
}

nvfp4_status moe_route_topk_ex(const float* logits, int32_t m, int32_t n_experts, int32_t top_k, int32_t flags,
                               const float* expert_scale, int32_t* ids, float* probs, int32_t* expert_offsets,
                               int32_t* sorted_pairs, cudaStream_t stream) {
  if (flags & ~kRouteSoftmaxAll) return NVFP4_ERR_SHAPE;
  if (expert_scale && !aligned(expert_scale, 4)) return NVFP4_ERR_ALIGN;
  if (!logits || !ids || !probs || !expert_offsets || !sorted_pairs) return NVFP4_ERR_NULL;
  if (m < 1 || m > 4096 || top_k < 1 || top_k > 32 || n_experts < top_k || n_experts > 1024 ||
      m * top_k > 16384)
    return NVFP4_ERR_SHAPE;
  if (!aligned(logits, 4) || !aligned(ids, 4) || !aligned(probs, 4) || !aligned(expert_offsets, 4) ||
      !aligned(sorted_pairs, 4))
    return NVFP4_ERR_ALIGN;
  const size_t smem = sizeof(int) * (static_cast<size_t>(m) * top_k + route_scratch(n_experts) + 32);
  const int nper = ceil_div(n_experts, 32);
  // a decode batch: one CTA; a larger batch: the top-k over many CTAs (one warp
  // per token), then the grouping by one CTA
  const bool split = m > 32;
  auto launch = [&](auto kernel, auto topk_kernel) -> nvfp4_status {
    if (!split) {
      if (set_smem(kernel, smem) != cudaSuccess) return NVFP4_ERR_CUDA;
      if (launch_pdl(kernel, dim3(1), dim3(kRouteThreads), smem, stream, logits, m, n_experts, top_k,
                     static_cast<int>(flags), expert_scale, ids, probs, expert_offsets, sorted_pairs) != cudaSuccess)
        return NVFP4_ERR_CUDA;
      return launched();
    }
    if (launch_pdl(topk_kernel, dim3(ceil_div(m, kTopkWarps)), dim3(kTopkWarps * 32), 0, stream, logits, m,
                   n_experts, top_k, static_cast<int>(flags), expert_scale, ids, probs) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    if (set_smem(moe_group_kernel, smem) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (launch_pdl(moe_group_kernel, dim3(1), dim3(kRouteThreads), smem, stream, static_cast<const int*>(ids),
                   m * top_k, n_experts, expert_offsets, sorted_pairs) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    return launched();
  };
  if (nper <= 1) return launch(moe_route_kernel<1>, moe_topk_kernel<1>);
  if (nper <= 2) return launch(moe_route_kernel<2>, moe_topk_kernel<2>);
  if (nper <= 4) return launch(moe_route_kernel<4>, moe_topk_kernel<4>);
  if (nper <= 8) return launch(moe_route_kernel<8>, moe_topk_kernel<8>);
  if (nper <= 16) return launch(moe_route_kernel<16>, moe_topk_kernel<16>);
  return launch(moe_route_kernel<32>, moe_topk_kernel<32>);
}

size_t moe_ffn_workspace_bytes(int32_t m, int32_t top_k, int32_t n_experts, int32_t d, int32_t inter) {
  if (m < 1 || m > 4096 || top_k < 1 || n_experts < top_k || m * top_k > 16384 || d < 64 || inter < 32) return 0;
  return moe_workspace(m, top_k, n_experts, d, inter, true).total;
}

}  // extern "C"

namespace nvfp4 {
namespace {

// The grouped FFN's argument checks (no launch).
nvfp4_status moe_ffn_check(const uint16_t* x, int32_t m, int32_t top_k, const float* probs,
                           const int32_t* expert_offsets, const int32_t* sorted_pairs, const nvfp4_weight* gate_up,
                           const nvfp4_weight* down, const nvfp4_weight* shared_gate_up,
                           const nvfp4_weight* shared_down, const uint16_t* out, const void* ws, size_t ws_bytes) {
  if (!x || !probs || !expert_offsets || !sorted_pairs || !out || !gate_up || !down) return NVFP4_ERR_NULL;
  if ((shared_gate_up == nullptr) != (shared_down == nullptr)) return NVFP4_ERR_NULL;
  const int n_exp = gate_up->num_matrices;
  if (n_exp < 1) return NVFP4_ERR_SHAPE;
  if (const nvfp4_status st = check_weight(gate_up, n_exp, NVFP4_GATED)) return st;
  if (const nvfp4_status st = check_weight(down, n_exp, 0)) return st;
  const int d = gate_up->k, inter = down->k;
  if (gate_up->n != 2 * inter || down->n != d) return NVFP4_ERR_SHAPE;
  const bool shared = shared_gate_up != nullptr;
  if (shared) {
    if (const nvfp4_status st = check_weight(shared_gate_up, 1, NVFP4_GATED)) return st;
    if (const nvfp4_status st = check_weight(shared_down, 1, 0)) return st;
    if (shared_gate_up->n != 2 * inter || shared_gate_up->k != d || shared_down->n != d || shared_down->k != inter)
      return NVFP4_ERR_SHAPE;
  }
  if (m < 1 || m > 4096 || top_k < 1 || top_k > n_exp || m * top_k > 16384 || (d % 64) || (inter % 64))
    return NVFP4_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(out, 4) || !aligned(probs, 4)) return NVFP4_ERR_ALIGN;
  if (!ws || ws_bytes < moe_ffn_workspace_bytes(m, top_k, n_exp, d, inter)) return NVFP4_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return NVFP4_ERR_ALIGN;
  return NVFP4_OK;
}

// The grouped FFN's launches (gate+up, down, combine) after moe_ffn_check.
nvfp4_status moe_ffn_launch(const uint16_t* x, int32_t m, int32_t top_k, const float* probs,
                            const int32_t* expert_offsets, const int32_t* sorted_pairs,
                            const nvfp4_weight* gate_up, const nvfp4_weight* down,
                            const nvfp4_weight* shared_gate_up, const nvfp4_weight* shared_down, uint16_t* out,
                            void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (const nvfp4_status st = moe_ffn_check(x, m, top_k, probs, expert_offsets, sorted_pairs, gate_up, down,
                                            shared_gate_up, shared_down, out, ws, ws_bytes))
    return st;
  const int n_exp = gate_up->num_matrices;
  const int d = gate_up->k, inter = down->k;
  const bool shared = shared_gate_up != nullptr;
  const MoESplits sp = moe_splits(m, top_k, n_exp, d, inter, true);
  const MoEWorkspace wl = moe_workspace(m, top_k, n_exp, d, inter, true);
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint16_t* h = reinterpret_cast<uint16_t*>(base + wl.fix);
  float* dpart = reinterpret_cast<float*>(base + wl.fix + wl.h);

  Job a{};
  a.w = static_cast<const uint8_t*>(gate_up->data);
  a.gs = gate_up->global_scale;
  a.w_sh = shared ? static_cast<const uint8_t*>(shared_gate_up->data) : nullptr;
  a.gs_sh = shared ? shared_gate_up->global_scale : nullptr;
  a.n = 2 * inter, a.k = d;
  a.ng = ceil_div(2 * inter, kGroupRows), a.kc = ceil_div(d, kTileK);
  a.x = x;
  a.m = m, a.n_experts = n_exp, a.top_k = top_k;
  a.offsets = expert_offsets, a.pairs = sorted_pairs;
  a.x_by_pair = 0;
  a.has_shared = shared;
  a.y = h, a.y_ld = inter;
  set_fixup(&a, base);
  Plan pa;
  if (!make_plan(m, sp.s_gu, a.ng, a.kc, sp.n_seg_max, n_exp, sp.per_run, false, std::max(1, sm_count()), &pa))
    return NVFP4_ERR_SHAPE;
  WeightMaps ma;
  if (!make_maps(gate_up, shared ? shared_gate_up : nullptr, &ma)) return NVFP4_ERR_CUDA;
  if (const nvfp4_status st = dispatch_stream<kEpiGated>(a, ma, pa, stream)) return st;

  Job b = a;
  b.w = static_cast<const uint8_t*>(down->data);
  b.gs = down->global_scale;
  b.w_sh = shared ? static_cast<const uint8_t*>(shared_down->data) : nullptr;
  b.gs_sh = shared ? shared_down->global_scale : nullptr;
  b.n = d, b.k = inter;
  b.ng = ceil_div(d, kGroupRows), b.kc = ceil_div(inter, kTileK);
  b.x = h;
  b.x_by_pair = 1;
  b.routing_ready = 1;  // the gate+up grid before it waited for the routing
  b.y = nullptr;
  b.yf = dpart, b.yf_ld = d;
  set_fixup(&b, base);
  Plan pb;
  if (!make_plan(m, sp.s_dn, b.ng, b.kc, sp.n_seg_max, n_exp, sp.per_run, true, std::max(1, sm_count()), &pb))
    return NVFP4_ERR_SHAPE;
  WeightMaps mb;
  if (!make_maps(down, shared ? shared_down : nullptr, &mb)) return NVFP4_ERR_CUDA;
  if (const nvfp4_status st = dispatch_stream<kEpiRows>(b, mb, pb, stream)) return st;

  const size_t total = static_cast<size_t>(m) * d;
  const int blocks = static_cast<int>(std::min<size_t>((total + 255) / 256, static_cast<size_t>(sm_count()) * 4));
  if (launch_pdl(moe_combine_kernel, dim3(std::max(1, blocks)), dim3(256), 0, stream, static_cast<const float*>(dpart),
                 probs, m, top_k, d, shared, out) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  return launched();
}

}  // namespace
}  // namespace nvfp4

extern "C" {

nvfp4_status moe_ffn_grouped(const uint16_t* x, int32_t m, int32_t top_k, const float* probs,
                             const int32_t* expert_offsets, const int32_t* sorted_pairs,
                             const nvfp4_weight* gate_up, const nvfp4_weight* down,
                             const nvfp4_weight* shared_gate_up, const nvfp4_weight* shared_down, uint16_t* out,
                             void* ws, size_t ws_bytes, cudaStream_t stream) {
  return moe_ffn_launch(x, m, top_k, probs, expert_offsets, sorted_pairs, gate_up, down, shared_gate_up, shared_down,
                        out, ws, ws_bytes, stream);
}

nvfp4_status moe_forward(const uint16_t* x, const float* logits, int32_t m, int32_t top_k, int32_t route_flags,
                         const float* expert_scale, int32_t* ids, float* probs, int32_t* expert_offsets,
                         int32_t* sorted_pairs, const nvfp4_weight* gate_up, const nvfp4_weight* down,
                         const nvfp4_weight* shared_gate_up, const nvfp4_weight* shared_down, uint16_t* out, void* ws,
                         size_t ws_bytes, cudaStream_t stream) {
  // both calls' arguments are checked before the first launch (the router's own
  // checks cover logits, ids, offsets and pairs; the FFN's the rest)
  if (!logits || !ids) return NVFP4_ERR_NULL;
  if (const nvfp4_status st = moe_ffn_check(x, m, top_k, probs, expert_offsets, sorted_pairs, gate_up, down,
                                            shared_gate_up, shared_down, out, ws, ws_bytes))
    return st;
  if (top_k > 32 || gate_up->num_matrices > 1024) return NVFP4_ERR_SHAPE;
  if (const nvfp4_status st = moe_route_topk_ex(logits, m, gate_up->num_matrices, top_k, route_flags, expert_scale,
                                                ids, probs, expert_offsets, sorted_pairs, stream))
    return st;
  return moe_ffn_launch(x, m, top_k, probs, expert_offsets, sorted_pairs, gate_up, down, shared_gate_up, shared_down,
                        out, ws, ws_bytes, stream);
}

}  // extern "C"

// ------------------------------------------------------------------ lm_head without allocation
// Scratch for lm_head_argmax_noalloc: the arrival counter and the per-token
// packed (value, row) maxima (4 KiB).  It lives in the library's own device
// memory, so callers pass only inputs and outputs.
namespace nvfp4 {
namespace {

constexpr size_t kNoAllocScratchBytes = kCounterBytes;
static __device__ __align__(256) uint8_t g_lm_head_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device.  The first call on a
// device looks it up (the host-side name of the array is not a device address)
// and zeroes it once; later calls reuse the cached address.
nvfp4_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_lm_head_scratch) != cudaSuccess || !ptr) return NVFP4_ERR_CUDA;
    if (cudaMemset(ptr, 0, kNoAllocScratchBytes) != cudaSuccess) return NVFP4_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

extern "C" nvfp4_status lm_head_argmax_noalloc(const nvfp4_weight* w, const uint16_t* x, int32_t m, float* max_logit,
                                               int32_t* argmax, cudaStream_t stream) {
  if (const nvfp4_status st = check_weight(w, 1, 0)) return st;
  if (!x || !max_logit || !argmax) return NVFP4_ERR_NULL;
  if (m < 1 || m > 16) return NVFP4_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(max_logit, 4) || !aligned(argmax, 4)) return NVFP4_ERR_ALIGN;
  if (lm_head_workspace_bytes(m, w->n) > kNoAllocScratchBytes) return NVFP4_ERR_WORKSPACE;
  void* ws = nullptr;
  if (const nvfp4_status st = scratch_address(&ws)) return st;
  // the arrival counter must read zero when the kernel starts
  if (cudaMemsetAsync(ws, 0, sizeof(unsigned), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  return lm_head_launch(w, x, m, max_logit, argmax, ws, stream);
}

// ------------------------------------------------------------------ plan query
namespace nvfp4 {
namespace {

// The plan a product would launch for these shapes on `sms` SMs.
bool product_plan(int product, int m, int n, int k, int top_k, int n_experts, int sms, Plan* pl) {
  const int ng = ceil_div(n, kGroupRows), kc = ceil_div(k, kTileK);
  switch (product) {
    case 0:  // dense GEMM
      if (m > 16) return false;
      return make_plan(m, dense_split(m, n, k), ng, kc, 1, 0, false, false, sms, pl);
    case 1:  // lm_head
      if (m > 16) return false;
      return make_plan(m, 1, ng, kc, 1, 0, false, false, sms, pl);
    case 2:    // MoE gate+up: n = 2 * inter, k = d
    case 3: {  // MoE down: n = d, k = inter
      if (top_k < 1 || n_experts < top_k || m > 4096 || m * top_k > 16384) return false;
      const int d = product == 2 ? k : n, inter = product == 2 ? n / 2 : k;
      const MoESplits sp = moe_splits(m, top_k, n_experts, d, inter, true);
      return make_plan(m, product == 2 ? sp.s_gu : sp.s_dn, ng, kc, sp.n_seg_max, n_experts, sp.per_run,
                       product == 3, sms, pl);
    }
    default:
      return false;
  }
}

}  // namespace
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_plan_info(int32_t product, int32_t m, int32_t n, int32_t k, int32_t top_k,
                                        int32_t n_experts, int32_t sms, int32_t* out, int32_t out_len) {
  if (!out) return NVFP4_ERR_NULL;
  if (out_len < 10 || sms < 1 || m < 1 || n < 1 || k < 16 || (k % 16)) return NVFP4_ERR_SHAPE;
  Plan pl;
  if (!product_plan(product, m, n, k, top_k, n_experts, sms, &pl)) return NVFP4_ERR_SHAPE;
  const int32_t v[11] = {pl.S,    pl.L,        pl.ns,           pl.xs_chunks, pl.xs_rows, pl.max_cta_segs,
                         pl.grid, pl.max_segs, pl.per_run ? 1 : 0, static_cast<int32_t>(pl.smem),
                         pl.slice_ctas ? 1 : 0};
  for (int i = 0; i < std::min<int32_t>(out_len, 11); ++i) out[i] = v[i];
  return NVFP4_OK;
}

// Walk a product's whole launch on the host with the kernels' own decomposition
// code (DecodeDeal / PrefillDeal) for n_seg segments.
extern "C" nvfp4_status nvfp4_plan_check(int32_t product, int32_t m, int32_t n, int32_t k, int32_t top_k,
                                         int32_t n_experts, int32_t sms, int32_t n_seg, int32_t* out,
                                         int32_t out_len) {
  if (!out) return NVFP4_ERR_NULL;
  if (out_len < 8 || sms < 1 || m < 1 || n < 1 || k < 16 || (k % 16) || n_seg < 1) return NVFP4_ERR_SHAPE;
  Plan pl;
  if (!product_plan(product, m, n, k, top_k, n_experts, sms, &pl)) return NVFP4_ERR_SHAPE;
  if (n_seg > pl.max_segs) return NVFP4_ERR_SHAPE;
  long long warp_max = 0, warp_sum = 0;  // (tile x chunk) steps per warp, decode kernel
  const int ng = ceil_div(n, kGroupRows), kc = ceil_div(k, kTileK);
  const long long cells = static_cast<long long>(n_seg) * ng * 4 * pl.S;  // (segment, group, tile, slice)
  if (cells > (1ll << 27)) return NVFP4_ERR_SHAPE;
  std::vector<uint8_t> seen(static_cast<size_t>(cells), 0);
  long long bad = 0, tiles = 0, pieces = 0;
  int max_span = 0, max_segs = 0;
  const long long counter_cells = static_cast<long long>(kFixCounterBytes / sizeof(unsigned));
  auto take = [&](const Piece& pc) {
    ++pieces;
    if (pc.tn < 1 || pc.t0 < 0 || pc.t0 + pc.tn > 4 || pc.seg < 0 || pc.seg >= n_seg || pc.grp < 0 || pc.grp >= ng ||
        pc.s < 0 || pc.s >= pl.S)
      return void(++bad);
    if (pl.S > 1 && (static_cast<long long>(pc.seg) * ng + pc.grp) * 4 + pc.t0 + pc.tn > counter_cells) ++bad;
    for (int t = pc.t0; t < pc.t0 + pc.tn; ++t) {
      const size_t c = ((static_cast<size_t>(pc.seg) * ng + pc.grp) * 4 + t) * pl.S + pc.s;
      if (seen[c]++) ++bad;
      ++tiles;
    }
  };
  if (!pl.per_run) {
    const DecodeDeal dd{n_seg, pl.S, pl.L, kc, ng, pl.grid, pl.slice_ctas ? 1 : 0};
    for (int b = 0; b < pl.grid; ++b) {
      int u0, u1, cseg0, nsc, c_lo, c_hi;
      dd.cta_range(b, u0, u1);
      dd.span(u0, u1, cseg0, nsc, c_lo, c_hi);
      max_span = std::max(max_span, c_hi - c_lo);
      max_segs = std::max(max_segs, nsc);
      for (int w = 0; w < kWarps; ++w) {
        long long work = 0;
        for (int j = 0; j < dd.n_pieces(u1 - u0, w); ++j) {
          const Piece pc = dd.piece(u0, u1 - u0, w, j);
          const int c0 = pc.s * pl.L, c1 = c0 + dd.slice_len(pc.s);
          if (c0 < c_lo || c1 > c_hi || pc.seg < cseg0 || pc.seg >= cseg0 + nsc) ++bad;  // inside the staged span
          take(pc);
          work += static_cast<long long>(pc.tn) * (c1 - c0);
        }
        warp_max = std::max(warp_max, work);
        warp_sum += work;
      }
    }
  } else {
    const PrefillDeal pd{n_seg, pl.S, pl.L, kc, ng, pl.grid};
    for (int b = 0; b < pl.grid; ++b) {
      int u0, u1;
      pd.cta_range(b, u0, u1);
      for (int r = 0; r < pd.n_runs(u0, u1); ++r) {
        const int lo = pd.run_lo(u0, r), hi = pd.run_hi(u0, u1, r);
        max_span = std::max(max_span, pd.slice_len(pd.run_slice(u0, r)));
        max_segs = std::max(max_segs, 1);
        for (int w = 0; w < kWarps; ++w)
          for (int j = 0; j < pd.n_pieces(hi - lo, w); ++j) {
            const Piece pc = pd.piece(lo, hi - lo, w, j);
            if (pc.seg != pd.run_seg(u0, r) || pc.s != pd.run_slice(u0, r)) ++bad;  // the run's block only
            take(pc);
          }
      }
    }
  }
  long long missing = 0;
  for (long long c = 0; c < cells; ++c) missing += seen[static_cast<size_t>(c)] == 0;
  out[0] = (bad == 0 && missing == 0) ? 1 : 0;
  out[1] = max_span;
  out[2] = pl.xs_chunks;
  out[3] = max_segs;
  out[4] = pl.max_cta_segs;
  out[5] = static_cast<int32_t>(std::min<long long>(tiles, 0x7FFFFFFF));
  out[6] = static_cast<int32_t>(std::min<long long>(pieces, 0x7FFFFFFF));
  out[7] = static_cast<int32_t>(pl.smem);
  if (out_len >= 10) {  // the busiest warp's (tile x chunk) steps and the mean over all warps, rounded up
    const long long warps = static_cast<long long>(pl.grid) * kWarps;
    out[8] = static_cast<int32_t>(std::min<long long>(warp_max, 0x7FFFFFFF));
    out[9] = static_cast<int32_t>(std::min<long long>((warp_sum + warps - 1) / warps, 0x7FFFFFFF));
  }
  return NVFP4_OK;
}
