// Router softmax + top-k: the step before the route layout.
//
// "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy), section
// Benchmark: the routes (INT32 expert ids, FP32 routing weights,
// renormalize=False) come from a router score / top-k computation over the
// router logits, which the page keeps outside its timed region.  Here:
// p = softmax(logits[t, :]) over all experts of the model; the k largest p in
// descending order, ties to the lower expert index; the weights are those p.
//
// One warp per token.  Lane l holds logits l, l + 32, ... in registers
// (at most 1024 experts).  The maximum and the sum of exp(l - max) are warp
// reductions in a fixed order (deterministic); each of the k rounds is a warp
// argmax over the not yet selected logits.  softmax is strictly increasing in
// the logit, so the selection compares the logits themselves, exactly.
#include <algorithm>

#include "common.cuh"
#include "router.cuh"

namespace w4a16 {

constexpr int kRouterThreads = 256;

// kPerLane: logits per lane held in registers (G <= 32 * kPerLane); the
// launcher picks the smallest power of two that covers G.
template <int kPerLane>
__global__ void __launch_bounds__(kRouterThreads) router_topk_kernel(const RouterParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (kRouterThreads / 32);
  const unsigned full = 0xFFFFFFFFu;
  const int per_lane = (p.G + 31) / 32;
  for (int t = blockIdx.x * (kRouterThreads / 32) + (threadIdx.x >> 5); t < p.T; t += warps) {
    const float* l = p.logits + static_cast<int64_t>(t) * p.G;
    float v[kPerLane];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int e = lane + 32 * i;
      v[i] = (i < per_lane && e < p.G) ? l[e] : -INFINITY;
      m = fmaxf(m, v[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(full, m, o));
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i)
      if (i < per_lane && lane + 32 * i < p.G) s += expf(v[i] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(full, s, o);
    uint32_t taken = 0;  // bit i: element i of this lane already selected
    for (int j = 0; j < p.k; ++j) {
      // this lane's best remaining (largest logit, lowest index on ties)
      float bv = -INFINITY;
      int be = 0x7FFFFFFF;
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) {
        const int e = lane + 32 * i;
        if (i < per_lane && e < p.G && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
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
      if (be < p.G && (be & 31) == lane) taken |= 1u << (be >> 5);
      if (lane == 0) {
        p.ids[static_cast<int64_t>(t) * p.k + j] = be;
        p.weights[static_cast<int64_t>(t) * p.k + j] = expf(bv - m) / s;
      }
    }
  }
}

cudaError_t launch_router(const RouterParams& p, int num_sms, cudaStream_t s, bool pdl) {
  const int warps_per_block = kRouterThreads / 32;
  const int grid = std::max(1, std::min((p.T + warps_per_block - 1) / warps_per_block, 8 * num_sms));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRouterThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int per_lane = (p.G + 31) / 32;
  if (per_lane <= 1) return cudaLaunchKernelEx(&cfg, router_topk_kernel<1>, p);
  if (per_lane <= 2) return cudaLaunchKernelEx(&cfg, router_topk_kernel<2>, p);
  if (per_lane <= 4) return cudaLaunchKernelEx(&cfg, router_topk_kernel<4>, p);
  if (per_lane <= 8) return cudaLaunchKernelEx(&cfg, router_topk_kernel<8>, p);
  if (per_lane <= 16) return cudaLaunchKernelEx(&cfg, router_topk_kernel<16>, p);
  return cudaLaunchKernelEx(&cfg, router_topk_kernel<32>, p);
}

}  // namespace w4a16
