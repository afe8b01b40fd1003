// Definitions behind dispatch_stream<kEpi> and epi_error_word<kEpi>, included
// by each epi_<name>.cu translation unit, which instantiates them for its
// epilogue only.
#pragma once

#include "launch.cuh"
#include "prefill.cuh"

namespace nvfp4 {

inline nvfp4_status launch_planned(void (*kernel)(Job, WeightMaps), Job p, const WeightMaps& maps, const Plan& plan,
                                   cudaStream_t stream) {
  if (set_smem(kernel, plan.smem) != cudaSuccess) return NVFP4_ERR_CUDA;
  p.S = plan.S;
  p.L = plan.L;
  p.ns = plan.ns;
  p.npre = kPreStages;
  p.slice_ctas = plan.slice_ctas ? 1 : 0;
  p.xs_chunks = plan.xs_chunks;
  p.xs_rows = plan.xs_rows;
  p.max_cta_segs = plan.max_cta_segs;
  p.max_segs = plan.max_segs;
  if (launch_pdl(kernel, dim3(plan.grid), dim3(kThreads), plan.smem, stream, p, maps) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  return launched();
}

template <int MT, bool kMMA, int kEpi>
nvfp4_status launch_stream(const Job& p, const WeightMaps& maps, const Plan& plan, cudaStream_t stream) {
  return launch_planned(stream_kernel<MT, kMMA, kEpi>, p, maps, plan, stream);
}

template <int kEpi>
nvfp4_status dispatch_stream(const Job& p, const WeightMaps& maps, const Plan& plan, cudaStream_t stream) {
  if constexpr (kEpi == kEpiGated || kEpi == kEpiRows)
    if (plan.per_run) return launch_planned(prefill_kernel<kEpi>, p, maps, plan, stream);
  // one token: CUDA cores with a warp-shuffle reduction; 2..8 tokens: one 8-slot
  // tensor-core column (empty slots read a zero row); 9..16: two columns
  if (p.m == 1) return launch_stream<1, false, kEpi>(p, maps, plan, stream);
  if (p.m <= 8) return launch_stream<8, true, kEpi>(p, maps, plan, stream);
  return launch_stream<16, true, kEpi>(p, maps, plan, stream);
}

template <int kEpi>
nvfp4_status epi_error_word(uint32_t* v, int clear) {
  unsigned w = 0;
  if (cudaMemcpyFromSymbol(&w, g_device_error, sizeof(w)) != cudaSuccess) return NVFP4_ERR_CUDA;
  *v = w;
  if (clear) {
    const unsigned z = 0;
    if (cudaMemcpyToSymbol(g_device_error, &z, sizeof(z)) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  return NVFP4_OK;
}

}  // namespace nvfp4
