// Host-side launch plumbing shared by the library's translation units: the
// launch plan, programmatic dependent launch, the shared-memory opt-in, and the
// per-epilogue launch entry points.  The streaming kernels are compiled in one
// translation unit per epilogue (epi_*.cu, compiled in parallel); the host
// unit (nvfp4_skinny.cu) reaches them through dispatch_stream<kEpi>.
#pragma once

#include <cstdlib>
#include <map>
#include <mutex>
#include <utility>

#include "kernel.cuh"

namespace nvfp4 {

constexpr size_t kMaxSmem = 227 * 1024;  // per-CTA opt-in limit on sm_103a
// Ring stages each warp fills before the wait for the previous grid (the rest
// follow the activation loads).
constexpr int kPreStages = 2;

struct Plan {
  int S, L, ns, xs_chunks, xs_rows, max_cta_segs, grid, max_segs;
  bool per_run;
  size_t smem;
  bool slice_ctas = false;  // single-segment job: CTA ranges aligned to K slices
};

inline nvfp4_status launched() { return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

// Allow the kernel the full opt-in shared memory, once per (kernel, device).
template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, bool> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
  std::lock_guard<std::mutex> lock(mu);
  if (done.count(key)) return bytes <= kMaxSmem ? cudaSuccess : cudaErrorInvalidValue;
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMaxSmem));
  if (e == cudaSuccess) done[key] = true;
  return e;
}

// Programmatic dependent launch (see kernel.cuh, "Launch overlap"); switched off
// by NVFP4_PDL=0 in the environment, for comparison runs.
inline bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("NVFP4_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The streaming kernel of epilogue kEpi for this job and plan (decode kernel
// specialised on m, or the prefill kernel for a plan with per-segment runs).
// Defined in epi_<name>.cu.
template <int kEpi>
nvfp4_status dispatch_stream(const Job& p, const WeightMaps& maps, const Plan& plan, cudaStream_t stream);

// The device error word of epilogue kEpi's translation unit: read into *v and
// cleared if `clear`.  Defined in epi_<name>.cu.
template <int kEpi>
nvfp4_status epi_error_word(uint32_t* v, int clear);

}  // namespace nvfp4
