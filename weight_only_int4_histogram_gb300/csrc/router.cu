// Router softmax + top-k: the step before the route layout.
//
// "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy), section
// Benchmark: the routes (INT32 expert ids, FP32 routing weights,
// renormalize=False) come from a router score / top-k computation over the
// router logits, which the page keeps outside its timed region.  Here:
// p = softmax(logits[t, :]) over all experts of the model; the k largest p in
// descending order, ties to the lower expert index; the weights are those p.
//
// One warp per token (warp_softmax_topk in router.cuh, shared with the fused
// router + route preparation of route_prep.cu).
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
  for (int t = blockIdx.x * (kRouterThreads / 32) + (threadIdx.x >> 5); t < p.T; t += warps) {
    int32_t* ids = p.ids + static_cast<int64_t>(t) * p.k;
    float* wts = p.weights + static_cast<int64_t>(t) * p.k;
    warp_softmax_topk<kPerLane>(p.logits + static_cast<int64_t>(t) * p.G, p.G, p.k, lane,
                                [&](int j, int id, float prob) {
                                  ids[j] = id;
                                  wts[j] = prob;
                                });
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
