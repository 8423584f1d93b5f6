// Router softmax + top-k launcher (router.cu), used by the C-ABI entry point.
#pragma once
#include <cstdint>

#include <cuda_runtime.h>
#include <math.h>

namespace w4a16 {

struct RouterParams {
  const float* logits;  // [T, G] FP32
  int32_t T, G, k;      // tokens, experts of the model (<= 1024), top-k (<= G)
  int32_t* ids;         // [T, k] out: expert index, descending probability
  float* weights;       // [T, k] out: softmax probability
};

cudaError_t launch_router(const RouterParams& p, int num_sms, cudaStream_t s, bool pdl);

#if defined(__CUDACC__)
// Softmax + top-k of one token's G logits by one warp: p = softmax(l) over all
// G experts; the k largest p in descending order, ties to the lower expert
// index.  Lane l holds logits l, l + 32, ... (kPerLane * 32 >= G) in registers;
// the maximum and the sum of exp(l - max) are warp reductions in a fixed order
// (deterministic); each of the k rounds is a warp argmax over the not yet
// selected logits.  softmax is strictly increasing in the logit, so the
// selection compares the logits themselves, exactly.  emit(j, id, prob) runs
// on lane 0 for every rank j = 0..k-1.
template <int kPerLane, typename Emit>
__device__ __forceinline__ void warp_softmax_topk(const float* l, int G, int k, int lane, Emit&& emit) {
  const unsigned full = 0xFFFFFFFFu;
  const int per_lane = (G + 31) / 32;
  float v[kPerLane];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    const int e = lane + 32 * i;
    v[i] = (i < per_lane && e < G) ? l[e] : -INFINITY;
    m = fmaxf(m, v[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(full, m, o));
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < kPerLane; ++i)
    if (i < per_lane && lane + 32 * i < G) s += expf(v[i] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(full, s, o);
  uint32_t taken = 0;  // bit i: element i of this lane already selected
  for (int j = 0; j < k; ++j) {
    // this lane's best remaining (largest logit, lowest index on ties)
    float bv = -INFINITY;
    int be = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int e = lane + 32 * i;
      if (i < per_lane && e < G && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(full, bv, o);
      const int oe = __shfl_xor_sync(full, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if (be < G && (be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == 0) emit(j, be, expf(bv - m) / s);
  }
}
#endif

}  // namespace w4a16
