// C-ABI entry points of the NVFP4 W4A16 skinny library (sm_103a).
// Host-side argument checks, launch geometry and kernel dispatch.  The kernels
// live in the included headers; everything is one translation unit.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "nvfp4_skinny.h"
#include "common.cuh"
#include "quant.cuh"
#include "gemm.cuh"
#include "moe.cuh"

namespace nvfp4 {

namespace {

constexpr size_t kCounterBytes = 4096;   // arrival counters at the start of a workspace
constexpr size_t kMaxSmem = 227 * 1024;  // per-CTA opt-in limit on sm_103a
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

nvfp4_status launched() { return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

nvfp4_status check_weight(const nvfp4_weight* w, int num_matrices, uint32_t flags) {
  if (!w || !w->data || !w->global_scale) return NVFP4_ERR_NULL;
  if (w->layout_version != NVFP4_LAYOUT_VERSION || w->flags != flags) return NVFP4_ERR_LAYOUT;
  if (w->n < 1 || w->k < 16 || (w->k % 16) || w->num_matrices != num_matrices) return NVFP4_ERR_SHAPE;
  if (!aligned(w->data, 16) || !aligned(w->global_scale, 4)) return NVFP4_ERR_ALIGN;
  return NVFP4_OK;
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

// ------------------------------------------------------------------ skinny launcher
struct Geometry {
  int csplit, ngroups, ns;
  size_t smem;
};

// Pick the k-split across CTAs and the ring depth for a dense or lm_head launch.
bool pick_geometry(bool mma, int slots, int nb, int kc, int m, bool allow_split, Geometry* out) {
  const int sms = sm_count();
  if (sms <= 0) return false;
  double best = 1e300;
  bool found = false;
  for (int c = 1; c <= (allow_split ? 8 : 1); c *= 2) {
    if (c > kc || sms / c < 1) break;
    const int ngroups = std::min(sms / c, nb);
    const int kcs_max = ceil_div(kc, c);
    int ns = 0;
    for (int s = 6; s >= 2; --s)
      if (skinny_smem_bytes(mma, slots, kcs_max, s) <= kMaxSmem) {
        ns = s;
        break;
      }
    if (!ns) continue;
    const double rb_per_group = ceil_div(nb, ngroups);
    const double est = rb_per_group * kcs_max * kTileBytes + double(kcs_max) * kTileK * slots * 2.0 +
                       (c > 1 ? double(c) * m * rb_per_group * 16 * 4 : 0.0);
    if (est < best) {
      best = est;
      *out = Geometry{c, ngroups, ns, skinny_smem_bytes(mma, slots, kcs_max, ns)};
      found = true;
    }
  }
  return found;
}

template <int MT, bool kMMA, int kEpi>
nvfp4_status launch_skinny(const SkinnyParams& p0, const Geometry& geo, cudaStream_t stream) {
  auto kernel = skinny_kernel<MT, kMMA, kEpi>;
  if (set_smem(kernel, geo.smem) != cudaSuccess) return NVFP4_ERR_CUDA;
  SkinnyParams p = p0;
  p.csplit = geo.csplit;
  p.ngroups = geo.ngroups;
  p.ns = geo.ns;
  kernel<<<geo.csplit * geo.ngroups, kThreads, geo.smem, stream>>>(p);
  return launched();
}

template <int kEpi>
nvfp4_status dispatch_skinny(const SkinnyParams& p, bool allow_split, cudaStream_t stream) {
  const bool mma = p.m >= 8;
  const int slots = mma ? (p.m <= 8 ? 8 : 16) : p.m;
  Geometry geo;
  if (!pick_geometry(mma, slots, p.nb, p.kc, p.m, allow_split, &geo)) return NVFP4_ERR_SHAPE;
  switch (p.m) {
    case 1: return launch_skinny<1, false, kEpi>(p, geo, stream);
    case 2: return launch_skinny<2, false, kEpi>(p, geo, stream);
    case 3: return launch_skinny<3, false, kEpi>(p, geo, stream);
    case 4: return launch_skinny<4, false, kEpi>(p, geo, stream);
    case 5: return launch_skinny<5, false, kEpi>(p, geo, stream);
    case 6: return launch_skinny<6, false, kEpi>(p, geo, stream);
    case 7: return launch_skinny<7, false, kEpi>(p, geo, stream);
    case 8: return launch_skinny<8, true, kEpi>(p, geo, stream);
    default: return launch_skinny<16, true, kEpi>(p, geo, stream);
  }
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

nvfp4_status nvfp4_device_error(uint32_t* out, int32_t clear) {
  if (!out) return NVFP4_ERR_NULL;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return NVFP4_ERR_CUDA;
  *out = v;
  if (clear) {
    const unsigned z = 0;
    if (cudaMemcpyToSymbol(g_device_error, &z, sizeof(z)) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  return NVFP4_OK;
}

size_t nvfp4_repacked_bytes(int32_t n, int32_t k, int32_t num_matrices) {
  if (n < 1 || k < 16 || (k % 16) || num_matrices < 1) return 0;
  const size_t nb = static_cast<size_t>(ceil_div(n, kTileRows));
  const size_t kc = static_cast<size_t>(ceil_div(k, kTileK));
  return static_cast<size_t>(num_matrices) * nb * kc * kTileBytes;
}

size_t nvfp4_quantize_workspace_bytes(int32_t num_matrices) {
  return num_matrices < 1 ? 0 : static_cast<size_t>(num_matrices) * sizeof(unsigned);
}

nvfp4_status nvfp4_quantize(const float* w, int32_t num_matrices, int32_t n, int32_t k, uint8_t* nibbles,
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
  quant_amax_kernel<<<dim3(bx, num_matrices), 256, 0, stream>>>(w, per, amax);
  if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  const size_t groups = per / 16;
  const int gx = static_cast<int>(std::min<size_t>((groups + 255) / 256, static_cast<size_t>(sms) * 8));
  quant_groups_kernel<<<dim3(gx, num_matrices), 256, 0, stream>>>(w, n, k, amax, nibbles, scales, global_scale);
  return launched();
}

nvfp4_status nvfp4_repack(const uint8_t* nibbles, const uint8_t* scales, int32_t num_matrices, int32_t n, int32_t k,
                          uint32_t flags, void* out, cudaStream_t stream) {
  if (!nibbles || !scales || !out) return NVFP4_ERR_NULL;
  if (num_matrices < 1 || n < 1 || k < 16 || (k % 16)) return NVFP4_ERR_SHAPE;
  if (flags & ~NVFP4_GATED) return NVFP4_ERR_LAYOUT;
  const bool gated = flags & NVFP4_GATED;
  if (gated && (n % 16)) return NVFP4_ERR_SHAPE;
  if (!aligned(out, 16)) return NVFP4_ERR_ALIGN;
  const int nb = ceil_div(n, kTileRows), kc = ceil_div(k, kTileK);
  const size_t tiles = static_cast<size_t>(num_matrices) * nb * kc;
  const int sms = std::max(1, sm_count());
  const int gx = static_cast<int>(std::min<size_t>((tiles * 36 + 255) / 256, static_cast<size_t>(sms) * 16));
  repack_kernel<<<gx, 256, 0, stream>>>(nibbles, scales, n, k, nb, kc, gated, tiles, static_cast<uint8_t*>(out));
  return launched();
}

size_t nvfp4_gemm_workspace_bytes(int32_t m, int32_t n, int32_t k) {
  if (m < 1 || m > 16 || n < 1 || k < 16) return 0;
  return kCounterBytes + static_cast<size_t>(8) * m * ceil_div(n, kTileRows) * kTileRows * sizeof(float);
}

nvfp4_status nvfp4_gemm(const nvfp4_weight* w, const uint16_t* x, int32_t m, uint16_t* y, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  if (const nvfp4_status st = check_weight(w, 1, 0)) return st;
  if (!x || !y) return NVFP4_ERR_NULL;
  if (m < 1 || m > 16) return NVFP4_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(y, 4)) return NVFP4_ERR_ALIGN;
  if (!ws || ws_bytes < nvfp4_gemm_workspace_bytes(m, w->n, w->k)) return NVFP4_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return NVFP4_ERR_ALIGN;
  SkinnyParams p{};
  p.w = static_cast<const uint8_t*>(w->data);
  p.gscale = w->global_scale;
  p.x = x;
  p.m = m, p.n = w->n, p.k = w->k;
  p.nb = ceil_div(w->n, kTileRows), p.kc = ceil_div(w->k, kTileK);
  p.y = y;
  p.counters = static_cast<unsigned*>(ws);
  p.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kCounterBytes);
  return dispatch_skinny<kEpiStore>(p, true, stream);
}

size_t lm_head_workspace_bytes(int32_t m, int32_t vocab) {
  if (m < 1 || m > 16 || vocab < 1) return 0;
  return kCounterBytes + static_cast<size_t>(1024) * m * (sizeof(float) + sizeof(int));
}

nvfp4_status lm_head_argmax(const nvfp4_weight* w, const uint16_t* x, int32_t m, float* max_logit, int32_t* argmax,
                            void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (const nvfp4_status st = check_weight(w, 1, 0)) return st;
  if (!x || !max_logit || !argmax) return NVFP4_ERR_NULL;
  if (m < 1 || m > 16) return NVFP4_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(max_logit, 4) || !aligned(argmax, 4)) return NVFP4_ERR_ALIGN;
  if (!ws || ws_bytes < lm_head_workspace_bytes(m, w->n)) return NVFP4_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return NVFP4_ERR_ALIGN;
  SkinnyParams p{};
  p.w = static_cast<const uint8_t*>(w->data);
  p.gscale = w->global_scale;
  p.x = x;
  p.m = m, p.n = w->n, p.k = w->k;
  p.nb = ceil_div(w->n, kTileRows), p.kc = ceil_div(w->k, kTileK);
  p.counters = static_cast<unsigned*>(ws);
  p.am_val = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kCounterBytes);
  p.am_idx = reinterpret_cast<int*>(p.am_val + 1024 * m);
  p.max_logit = max_logit;
  p.argmax = argmax;
  return dispatch_skinny<kEpiArgmax>(p, false, stream);
}

}  // extern "C"

// ------------------------------------------------------------------ MoE
namespace nvfp4 {
namespace {

size_t align16(size_t b) { return (b + 15) & ~static_cast<size_t>(15); }

template <int MT, bool kMMA, int kEpi>
nvfp4_status launch_moe(MoEParams p, cudaStream_t stream) {
  const int slots = kMMA ? ((MT + 7) / 8) * 8 : MT;
  int ns = 0;
  for (int s = 6; s >= 2; --s)
    if (moe_smem_bytes(kMMA, slots, p.kc, s, p.n_experts) <= kMaxSmem) {
      ns = s;
      break;
    }
  if (!ns) return NVFP4_ERR_SHAPE;
  p.ns = ns;
  const size_t smem = moe_smem_bytes(kMMA, slots, p.kc, ns, p.n_experts);
  auto kernel = moe_ffn_kernel<MT, kMMA, kEpi>;
  if (set_smem(kernel, smem) != cudaSuccess) return NVFP4_ERR_CUDA;
  kernel<<<std::max(1, sm_count()), kThreads, smem, stream>>>(p);
  return launched();
}

template <int kEpi>
nvfp4_status dispatch_moe(const MoEParams& p, cudaStream_t stream) {
  if (p.m == 1) return launch_moe<1, false, kEpi>(p, stream);
  if (p.m <= 8) return launch_moe<8, true, kEpi>(p, stream);
  return launch_moe<16, true, kEpi>(p, stream);
}

}  // namespace
}  // namespace nvfp4

extern "C" {

nvfp4_status moe_route_topk(const float* logits, int32_t m, int32_t n_experts, int32_t top_k, int32_t* ids,
                            float* probs, int32_t* expert_offsets, int32_t* sorted_pairs, cudaStream_t stream) {
  if (!logits || !ids || !probs || !expert_offsets || !sorted_pairs) return NVFP4_ERR_NULL;
  if (m < 1 || m > 4096 || top_k < 1 || top_k > 32 || n_experts < top_k || n_experts > 1024 ||
      m * top_k > 16384)
    return NVFP4_ERR_SHAPE;
  if (!aligned(logits, 4) || !aligned(ids, 4) || !aligned(probs, 4) || !aligned(expert_offsets, 4) ||
      !aligned(sorted_pairs, 4))
    return NVFP4_ERR_ALIGN;
  const size_t smem = sizeof(int) * (static_cast<size_t>(m) * top_k + n_experts + 1);
  if (set_smem(moe_route_kernel, smem) != cudaSuccess) return NVFP4_ERR_CUDA;
  moe_route_kernel<<<1, kRouteThreads, smem, stream>>>(logits, m, n_experts, top_k, ids, probs, expert_offsets,
                                                        sorted_pairs);
  return launched();
}

size_t moe_ffn_workspace_bytes(int32_t m, int32_t top_k, int32_t d, int32_t inter) {
  if (m < 1 || top_k < 1 || d < 1 || inter < 1) return 0;
  const size_t pairs = static_cast<size_t>(m) * top_k + m;
  return align16(pairs * inter * sizeof(uint16_t)) + pairs * d * sizeof(float);
}

nvfp4_status moe_ffn_grouped(const uint16_t* x, int32_t m, int32_t top_k, const float* probs,
                             const int32_t* expert_offsets, const int32_t* sorted_pairs,
                             const nvfp4_weight* gate_up, const nvfp4_weight* down,
                             const nvfp4_weight* shared_gate_up, const nvfp4_weight* shared_down, uint16_t* out,
                             void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!x || !probs || !expert_offsets || !sorted_pairs || !out || !gate_up || !down) return NVFP4_ERR_NULL;
  if ((shared_gate_up == nullptr) != (shared_down == nullptr)) return NVFP4_ERR_NULL;
  const int n_exp = gate_up->num_matrices;
  if (n_exp < 1) return NVFP4_ERR_SHAPE;
  if (const nvfp4_status st = check_weight(gate_up, n_exp, NVFP4_GATED)) return st;
  if (const nvfp4_status st = check_weight(down, n_exp, 0)) return st;
  const int d = gate_up->k, inter = down->k;
  if (gate_up->n != 2 * inter || down->n != d) return NVFP4_ERR_SHAPE;
  if (shared_gate_up) {
    if (const nvfp4_status st = check_weight(shared_gate_up, 1, NVFP4_GATED)) return st;
    if (const nvfp4_status st = check_weight(shared_down, 1, 0)) return st;
    if (shared_gate_up->n != 2 * inter || shared_gate_up->k != d || shared_down->n != d || shared_down->k != inter)
      return NVFP4_ERR_SHAPE;
  }
  if (m < 1 || m > 16 || top_k < 1 || top_k > n_exp || (d % 64) || (inter % 64)) return NVFP4_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(out, 4) || !aligned(probs, 4)) return NVFP4_ERR_ALIGN;
  if (!ws || ws_bytes < moe_ffn_workspace_bytes(m, top_k, d, inter)) return NVFP4_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return NVFP4_ERR_ALIGN;
  const size_t pairs_total = static_cast<size_t>(m) * top_k + m;
  uint16_t* h = static_cast<uint16_t*>(ws);
  float* dpart = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + align16(pairs_total * inter * sizeof(uint16_t)));

  MoEParams a{};
  a.w = static_cast<const uint8_t*>(gate_up->data);
  a.gs = gate_up->global_scale;
  a.w_sh = shared_gate_up ? static_cast<const uint8_t*>(shared_gate_up->data) : nullptr;
  a.gs_sh = shared_gate_up ? shared_gate_up->global_scale : nullptr;
  a.mat_bytes = nvfp4_repacked_bytes(2 * inter, d, 1);
  a.x = x;
  a.k = d;
  a.nb = ceil_div(2 * inter, kTileRows);
  a.kc = ceil_div(d, kTileK);
  a.m = m, a.top_k = top_k, a.n_experts = n_exp;
  a.offsets = expert_offsets, a.pairs = sorted_pairs;
  a.h_out = h;
  a.out_cols = inter;
  if (const nvfp4_status st = dispatch_moe<kEpiGatedGelu>(a, stream)) return st;

  MoEParams b = a;
  b.w = static_cast<const uint8_t*>(down->data);
  b.gs = down->global_scale;
  b.w_sh = shared_down ? static_cast<const uint8_t*>(shared_down->data) : nullptr;
  b.gs_sh = shared_down ? shared_down->global_scale : nullptr;
  b.mat_bytes = nvfp4_repacked_bytes(d, inter, 1);
  b.x = h;
  b.k = inter;
  b.nb = ceil_div(d, kTileRows);
  b.kc = ceil_div(inter, kTileK);
  b.h_out = nullptr;
  b.d_out = dpart;
  b.out_cols = d;
  if (const nvfp4_status st = dispatch_moe<kEpiPartial>(b, stream)) return st;

  const size_t total = static_cast<size_t>(m) * d;
  const int blocks = static_cast<int>(std::min<size_t>((total + 255) / 256, static_cast<size_t>(sm_count()) * 4));
  moe_combine_kernel<<<std::max(1, blocks), 256, 0, stream>>>(dpart, probs, m, top_k, d, shared_gate_up != nullptr,
                                                               out);
  return launched();
}

}  // extern "C"

// ------------------------------------------------------------------ lm_head without allocation
// Scratch for lm_head_argmax_noalloc: the arrival counter (first 4 KiB) and the
// per-CTA (value, row) partials for up to 1024 CTAs x 16 tokens.  It lives in
// the library's own device memory, so callers pass only inputs and outputs.
namespace nvfp4 {
namespace {

constexpr size_t kNoAllocScratchBytes = kCounterBytes + static_cast<size_t>(1024) * 16 * (sizeof(float) + sizeof(int));
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
  SkinnyParams p{};
  p.w = static_cast<const uint8_t*>(w->data);
  p.gscale = w->global_scale;
  p.x = x;
  p.m = m, p.n = w->n, p.k = w->k;
  p.nb = ceil_div(w->n, kTileRows), p.kc = ceil_div(w->k, kTileK);
  p.counters = static_cast<unsigned*>(ws);
  p.am_val = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kCounterBytes);
  p.am_idx = reinterpret_cast<int*>(p.am_val + 1024 * m);
  p.max_logit = max_logit;
  p.argmax = argmax;
  return dispatch_skinny<kEpiArgmax>(p, false, stream);
}
