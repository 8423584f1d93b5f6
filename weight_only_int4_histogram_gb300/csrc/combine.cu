// Top-k weighted combine of the per-route expert outputs.
//
// "perf: reduce split W4A16 routing and output overhead" (FlashInfer),
// section Description: expert outputs are stored to scratch, then combined in
// FP32 in fixed top-k order before one cast of the output, with no atomic or
// TMA reduction.  "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy),
// section Benchmark: the weighted reduction closes the timed forward.
//
// Expert outputs arrive in the activation dtype (the FlashInfer page's 16-bit
// scratch) or, when the down GEMM ran split-K, as FP32 split partials.  One
// thread owns four consecutive output columns of one token, so the reduction
// order is fixed by construction: split partials s = 0..S-1 of a route are
// summed first, then routes j = 0..k-1 are accumulated as
// acc = acc + w'[j] * y (two roundings, no contraction); invalid routes are
// skipped.  Bitwise deterministic.
#include "common.cuh"

namespace w4a16 {

template <int DT>
__device__ __forceinline__ uint16_t to_bits(float f) {
  if (DT == DT_BF16) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
  } else {
    __half h = __float2half_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
  }
}

template <int DT>
__device__ __forceinline__ float from_bits(uint32_t b) {
  if (DT == DT_BF16) return __uint_as_float(b << 16);
  __half h;
  *reinterpret_cast<uint16_t*>(&h) = static_cast<uint16_t>(b);
  return __half2float(h);
}

// Four consecutive expert-output values of one route (split partials summed in order).
template <int DT, bool Y16>
__device__ __forceinline__ float4 load_y(const CombineParams& p, int slot, int c) {
  const int64_t off = static_cast<int64_t>(slot) * p.H + c;
  if (Y16) {
    const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.y) + off);
    return make_float4(from_bits<DT>(u.x & 0xFFFFu), from_bits<DT>(u.x >> 16), from_bits<DT>(u.y & 0xFFFFu),
                       from_bits<DT>(u.y >> 16));
  }
  const float* ys = reinterpret_cast<const float*>(p.y) + off;
  float4 y = *reinterpret_cast<const float4*>(ys);
  for (int s = 1; s < p.splits; ++s) {
    const float4 z = *reinterpret_cast<const float4*>(ys + static_cast<int64_t>(s) * p.slots_cap * p.H);
    y.x = __fadd_rn(y.x, z.x);
    y.y = __fadd_rn(y.y, z.y);
    y.z = __fadd_rn(y.z, z.z);
    y.w = __fadd_rn(y.w, z.w);
  }
  return y;
}

template <int DT, bool Y16>
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p) {
  pdl_wait();
  pdl_launch_dependents();
  // the fused expert launch's queue state, reset for a forward that reuses
  // this route layout (that launch has completed: pdl_wait)
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < p.zero_len; i += blockDim.x) p.zero[i] = 0;
  const int t = blockIdx.x;
  const int c = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
  if (c >= p.H) return;
  const int k = p.k;
  const float* tw = p.topk_weights + static_cast<int64_t>(t) * k;
  const int32_t* inv = p.inv + static_cast<int64_t>(t) * k;
  float wsum = 0.0f;
  if (p.renormalize) {
    for (int j = 0; j < k; ++j) wsum = __fadd_rn(wsum, tw[j]);
  }
  float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
  for (int j = 0; j < k; ++j) {
    const int slot = inv[j];
    if (slot < 0) continue;
    float w = tw[j];
    if (p.renormalize) w = (wsum != 0.0f) ? __fdiv_rn(w, wsum) : 0.0f;
    const float4 y = load_y<DT, Y16>(p, slot, c);
    a0 = __fadd_rn(a0, __fmul_rn(w, y.x));
    a1 = __fadd_rn(a1, __fmul_rn(w, y.y));
    a2 = __fadd_rn(a2, __fmul_rn(w, y.z));
    a3 = __fadd_rn(a3, __fmul_rn(w, y.w));
  }
  uint2 o;
  o.x = static_cast<uint32_t>(to_bits<DT>(a0)) | (static_cast<uint32_t>(to_bits<DT>(a1)) << 16);
  o.y = static_cast<uint32_t>(to_bits<DT>(a2)) | (static_cast<uint32_t>(to_bits<DT>(a3)) << 16);
  *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.out) + static_cast<int64_t>(t) * p.H + c) = o;
}

cudaError_t launch_combine(int dtype, const CombineParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  const int threads = 256;
  cfg.gridDim = dim3(p.T, (p.H / 4 + threads - 1) / threads);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (dtype == DT_BF16)
    return p.y16 ? cudaLaunchKernelEx(&cfg, combine_kernel<DT_BF16, true>, p)
                 : cudaLaunchKernelEx(&cfg, combine_kernel<DT_BF16, false>, p);
  return p.y16 ? cudaLaunchKernelEx(&cfg, combine_kernel<DT_FP16, true>, p)
               : cudaLaunchKernelEx(&cfg, combine_kernel<DT_FP16, false>, p);
}

}  // namespace w4a16
