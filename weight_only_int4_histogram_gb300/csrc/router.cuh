// Router softmax + top-k launcher (router.cu), used by the C-ABI entry point.
#pragma once
#include <cstdint>

#include <cuda_runtime.h>

namespace w4a16 {

struct RouterParams {
  const float* logits;  // [T, G] FP32
  int32_t T, G, k;      // tokens, experts of the model (<= 1024), top-k (<= G)
  int32_t* ids;         // [T, k] out: expert index, descending probability
  float* weights;       // [T, k] out: softmax probability
};

cudaError_t launch_router(const RouterParams& p, int num_sms, cudaStream_t s, bool pdl);

}  // namespace w4a16
