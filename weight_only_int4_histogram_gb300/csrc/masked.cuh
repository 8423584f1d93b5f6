// Masked-count layout launchers (route_prep.cu), used by the C-ABI entry point.
#pragma once
#include <cstdint>

#include <cuda_runtime.h>

namespace w4a16 {

// Routes of the masked-count layout: row r = e * max_rows + i of the
// expert-major activations becomes one token with a single route, to global
// expert expert_offset + e with weight 1 when i < clamp(counts[e], 0,
// max_rows), else an invalid route (-1).
cudaError_t launch_masked_routes(const int32_t* counts, int32_t E, int32_t max_rows, int32_t expert_offset,
                                 int32_t* ids, float* weights, int num_sms, cudaStream_t s, bool pdl);

// Rows i >= min(counts[e], max_rows) of out [E][max_rows][H] (16-bit
// elements, H a multiple of 8) set to +0; counts are route preparation's
// per-expert route counts.
cudaError_t launch_masked_zero_rows(const int32_t* counts, int32_t E, int32_t max_rows, int32_t H, void* out,
                                    cudaStream_t s, bool pdl);

}  // namespace w4a16
