// The streaming kernels of the sample epilogue (kEpiSample): one translation unit per
// epilogue so that the library's kernels compile in parallel.
#include "epilogue.cuh"

namespace nvfp4 {
template nvfp4_status dispatch_stream<kEpiSample>(const Job&, const WeightMaps&, const Plan&, cudaStream_t);
template nvfp4_status epi_error_word<kEpiSample>(uint32_t*, int);
}  // namespace nvfp4
