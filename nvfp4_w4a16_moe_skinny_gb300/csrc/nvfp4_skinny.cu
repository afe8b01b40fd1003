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
#include "kernel.cuh"
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

// ------------------------------------------------------------------ streaming-kernel plans
// The K split S is chosen from the shapes alone, against a fixed reference
// parallelism (152 SMs x 16 warps), so workspace sizes are host-computable and
// identical on every device; the grid is the device's SM count.
constexpr int kPlanSMs = 152;
constexpr int kMaxSplit = 16;

struct Plan {
  int S, L, ns, xs_chunks;
  size_t smem;
};

int nacc_per_lane(int m) { return m <= 7 ? 4 * m * 2 : (m <= 8 ? 16 : 32); }
bool use_mma(int m) { return m >= 8; }
int slots_of(int m) { return use_mma(m) ? (m <= 8 ? 8 : 16) : m; }

// S for `pieces1` (segments x groups) unsplit pieces of kc chunks each.
int choose_split(long long pieces1, int kc, bool mma) {
  const long long warps = static_cast<long long>(kPlanSMs) * kWarps;
  if (pieces1 >= warps) return 1;
  // shortest slice worth a fixup partial: a partial costs a fence and 1-4 KiB
  // through L2, against 2,304 B of weights per chunk
  const int lmin = mma ? 8 : 4;
  int s = static_cast<int>((warps + pieces1 - 1) / pieces1);
  s = std::min(s, std::max(1, kc / lmin));
  s = std::min(s, kMaxSplit);
  const int L = ceil_div(kc, s);
  return ceil_div(kc, L);
}

bool make_plan(int m, int S, int ng, int kc, int n_seg_max, int n_experts, Plan* out) {
  const int sms = std::max(1, sm_count());
  const bool mma = use_mma(m);
  const int slots = slots_of(m);
  const int L = ceil_div(kc, S);
  int xs_chunks = kc;
  if (S > 1) {
    const long long pc = (static_cast<long long>(n_seg_max) * S * ng + sms - 1) / sms;
    xs_chunks = static_cast<int>(std::min<long long>(kc, ((pc + ng - 1) / ng + 1) * L));
  }
  for (int ns = 8; ns >= 2; --ns) {
    const size_t smem = stream_smem_bytes(mma, slots, xs_chunks, ns, n_experts);
    if (smem <= kMaxSmem) {
      *out = Plan{S, L, ns, xs_chunks, smem};
      return true;
    }
  }
  return false;
}

template <int MT, bool kMMA, int kEpi>
nvfp4_status launch_stream(Job p, const Plan& plan, cudaStream_t stream) {
  auto kernel = stream_kernel<MT, kMMA, kEpi>;
  if (set_smem(kernel, plan.smem) != cudaSuccess) return NVFP4_ERR_CUDA;
  p.S = plan.S;
  p.L = plan.L;
  p.ns = plan.ns;
  p.xs_chunks = plan.xs_chunks;
  kernel<<<std::max(1, sm_count()), kThreads, plan.smem, stream>>>(p);
  return launched();
}

template <int kEpi>
nvfp4_status dispatch_stream(const Job& p, const Plan& plan, cudaStream_t stream) {
  switch (p.m) {
    case 1: return launch_stream<1, false, kEpi>(p, plan, stream);
    case 2: return launch_stream<2, false, kEpi>(p, plan, stream);
    case 3: return launch_stream<3, false, kEpi>(p, plan, stream);
    case 4: return launch_stream<4, false, kEpi>(p, plan, stream);
    case 5: return launch_stream<5, false, kEpi>(p, plan, stream);
    case 6: return launch_stream<6, false, kEpi>(p, plan, stream);
    case 7: return launch_stream<7, false, kEpi>(p, plan, stream);
    case 8: return launch_stream<8, true, kEpi>(p, plan, stream);
    default: return launch_stream<16, true, kEpi>(p, plan, stream);
  }
}

// A fixup area is a fixed 64 KiB of arrival counters (one per segment x group,
// at most 16,384) followed by the partials.  The counters sit at the same place
// whatever the shape, and every call leaves them zero, so one zero-filled
// workspace can serve calls of different shapes.
constexpr size_t kFixCounterBytes = 64 * 1024;

size_t fixup_bytes(int m, int S, int ng, int n_seg_max) {
  if (S <= 1) return 0;
  return kFixCounterBytes + static_cast<size_t>(n_seg_max) * ng * S * 32 * nacc_per_lane(m) * sizeof(float);
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
  return choose_split(ceil_div(n, kGroupRows), ceil_div(k, kTileK), use_mma(m));
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
  const size_t nb = static_cast<size_t>(ceil_div(n, kGroupRows)) * (kGroupRows / kTileRows);
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
  if (gated && (n % kGroupRows)) return NVFP4_ERR_SHAPE;
  if (!aligned(out, 16)) return NVFP4_ERR_ALIGN;
  const int ng = ceil_div(n, kGroupRows), kc = ceil_div(k, kTileK);
  const size_t tiles = static_cast<size_t>(num_matrices) * ng * kc * 4;
  const int sms = std::max(1, sm_count());
  const int gx = static_cast<int>(std::min<size_t>((tiles * 36 + 255) / 256, static_cast<size_t>(sms) * 16));
  repack_kernel<<<gx, 256, 0, stream>>>(nibbles, scales, n, k, ng, kc, gated, tiles, static_cast<uint8_t*>(out));
  return launched();
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
  if (!make_plan(m, dense_split(m, w->n, w->k), p.ng, p.kc, 1, 0, &plan)) return NVFP4_ERR_SHAPE;
  return dispatch_stream<kEpiStore>(p, plan, stream);
}

size_t lm_head_workspace_bytes(int32_t m, int32_t vocab) {
  if (m < 1 || m > 16 || vocab < 1) return 0;
  return kCounterBytes + static_cast<size_t>(1024) * m * (sizeof(float) + sizeof(int));
}

}  // extern "C"

namespace nvfp4 {
namespace {

// The lm_head never splits K: a split would put partial logits in memory.
nvfp4_status lm_head_launch(const nvfp4_weight* w, const uint16_t* x, int32_t m, float* max_logit, int32_t* argmax,
                            void* ws, cudaStream_t stream) {
  Job p = dense_job(w, x, m);
  p.am_cnt = static_cast<unsigned*>(ws);
  p.am_val = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kCounterBytes);
  p.am_idx = reinterpret_cast<int*>(p.am_val + 1024 * m);
  p.max_logit = max_logit;
  p.argmax = argmax;
  Plan plan;
  if (!make_plan(m, 1, p.ng, p.kc, 1, 0, &plan)) return NVFP4_ERR_SHAPE;
  return dispatch_stream<kEpiArgmax>(p, plan, stream);
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
  if (sm_count() > 1024) return NVFP4_ERR_SHAPE;
  return lm_head_launch(w, x, m, max_logit, argmax, ws, stream);
}

}  // extern "C"

// ------------------------------------------------------------------ MoE
namespace nvfp4 {
namespace {

size_t align16(size_t b) { return (b + 15) & ~static_cast<size_t>(15); }

// Expected number of experts that receive at least one of the m*top_k pairs
// (uniform routing), plus the shared expert: the planning estimate of segments.
int expected_segments(int m, int top_k, int n_experts, bool shared) {
  double miss = 1.0;
  for (int t = 0; t < m; ++t) miss *= 1.0 - static_cast<double>(top_k) / n_experts;
  const int est = static_cast<int>(n_experts * (1.0 - miss) + 0.5);
  return std::max(1, std::min(est, n_experts)) + (shared ? 1 : 0);
}

struct MoESplits {
  int s_gu, s_dn, n_seg_max;
};

MoESplits moe_splits(int m, int top_k, int n_experts, int d, int inter, bool shared) {
  const int n_seg_est = expected_segments(m, top_k, n_experts, shared);
  MoESplits r;
  r.s_gu = choose_split(static_cast<long long>(n_seg_est) * ceil_div(2 * inter, kGroupRows), ceil_div(d, kTileK),
                        use_mma(m));
  r.s_dn = choose_split(static_cast<long long>(n_seg_est) * ceil_div(d, kGroupRows), ceil_div(inter, kTileK),
                        use_mma(m));
  r.n_seg_max = std::min(n_experts, m * top_k) + (shared ? 1 : 0);
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
  // gate_up and down share one fixup area: the down launch starts after gate_up ends
  w.fix = align16(std::max(fixup_bytes(m, sp.s_gu, ceil_div(2 * inter, kGroupRows), sp.n_seg_max),
                           fixup_bytes(m, sp.s_dn, ceil_div(d, kGroupRows), sp.n_seg_max)));
  w.total = w.h + w.d + w.fix;
  return w;
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

size_t moe_ffn_workspace_bytes(int32_t m, int32_t top_k, int32_t n_experts, int32_t d, int32_t inter) {
  if (m < 1 || m > 16 || top_k < 1 || n_experts < top_k || d < 64 || inter < 32) return 0;
  return moe_workspace(m, top_k, n_experts, d, inter, true).total;
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
  const bool shared = shared_gate_up != nullptr;
  if (shared) {
    if (const nvfp4_status st = check_weight(shared_gate_up, 1, NVFP4_GATED)) return st;
    if (const nvfp4_status st = check_weight(shared_down, 1, 0)) return st;
    if (shared_gate_up->n != 2 * inter || shared_gate_up->k != d || shared_down->n != d || shared_down->k != inter)
      return NVFP4_ERR_SHAPE;
  }
  if (m < 1 || m > 16 || top_k < 1 || top_k > n_exp || (d % 64) || (inter % 64)) return NVFP4_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(out, 4) || !aligned(probs, 4)) return NVFP4_ERR_ALIGN;
  if (!ws || ws_bytes < moe_ffn_workspace_bytes(m, top_k, n_exp, d, inter)) return NVFP4_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return NVFP4_ERR_ALIGN;
  const MoESplits sp = moe_splits(m, top_k, n_exp, d, inter, true);
  const MoEWorkspace wl = moe_workspace(m, top_k, n_exp, d, inter, true);
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint16_t* h = reinterpret_cast<uint16_t*>(base);
  float* dpart = reinterpret_cast<float*>(base + wl.h);

  Job a{};
  a.w = static_cast<const uint8_t*>(gate_up->data);
  a.gs = gate_up->global_scale;
  a.w_sh = shared ? static_cast<const uint8_t*>(shared_gate_up->data) : nullptr;
  a.gs_sh = shared ? shared_gate_up->global_scale : nullptr;
  a.mat_bytes = nvfp4_repacked_bytes(2 * inter, d, 1);
  a.n = 2 * inter, a.k = d;
  a.ng = ceil_div(2 * inter, kGroupRows), a.kc = ceil_div(d, kTileK);
  a.x = x;
  a.m = m, a.n_experts = n_exp, a.top_k = top_k;
  a.offsets = expert_offsets, a.pairs = sorted_pairs;
  a.x_by_pair = 0;
  a.has_shared = shared;
  a.y = h, a.y_ld = inter;
  set_fixup(&a, base + wl.h + wl.d);
  Plan pa;
  if (!make_plan(m, sp.s_gu, a.ng, a.kc, sp.n_seg_max, n_exp, &pa)) return NVFP4_ERR_SHAPE;
  if (const nvfp4_status st = dispatch_stream<kEpiGated>(a, pa, stream)) return st;

  Job b = a;
  b.w = static_cast<const uint8_t*>(down->data);
  b.gs = down->global_scale;
  b.w_sh = shared ? static_cast<const uint8_t*>(shared_down->data) : nullptr;
  b.gs_sh = shared ? shared_down->global_scale : nullptr;
  b.mat_bytes = nvfp4_repacked_bytes(d, inter, 1);
  b.n = d, b.k = inter;
  b.ng = ceil_div(d, kGroupRows), b.kc = ceil_div(inter, kTileK);
  b.x = h;
  b.x_by_pair = 1;
  b.y = nullptr;
  b.yf = dpart, b.yf_ld = d;
  set_fixup(&b, base + wl.h + wl.d);
  Plan pb;
  if (!make_plan(m, sp.s_dn, b.ng, b.kc, sp.n_seg_max, n_exp, &pb)) return NVFP4_ERR_SHAPE;
  if (const nvfp4_status st = dispatch_stream<kEpiRows>(b, pb, stream)) return st;

  const size_t total = static_cast<size_t>(m) * d;
  const int blocks = static_cast<int>(std::min<size_t>((total + 255) / 256, static_cast<size_t>(sm_count()) * 4));
  moe_combine_kernel<<<std::max(1, blocks), 256, 0, stream>>>(dpart, probs, m, top_k, d, shared, out);
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
  if (lm_head_workspace_bytes(m, w->n) > kNoAllocScratchBytes || sm_count() > 1024) return NVFP4_ERR_WORKSPACE;
  void* ws = nullptr;
  if (const nvfp4_status st = scratch_address(&ws)) return st;
  // the arrival counter must read zero when the kernel starts
  if (cudaMemsetAsync(ws, 0, sizeof(unsigned), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  return lm_head_launch(w, x, m, max_logit, argmax, ws, stream);
}
