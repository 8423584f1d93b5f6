// Route-layout preparation ("histogram") for the local W4A16 MoE forward.
//
// Follows "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy),
// sections Benchmark (route preparation is part of the timed forward) and
// Modification (invalid routes and masked expert counts), and "perf: reduce
// split W4A16 routing and output overhead" (FlashInfer), section Description
// (routing-side bookkeeping on the route tiles).
//
// One CTA of 32 warps.  The flat routes r = t*k + j are cut into 32 contiguous
// chunks, one per warp, so "earlier warp" means "smaller flat index":
//   pass 1  per-warp histograms hist[w][e]: counts only, so shared-memory
//           integer atomics (exact, order-independent) suffice;
//   pass 2  column prefix over warps (routes of expert e in earlier chunks),
//           then a warp-shuffle exclusive scan over experts of the padded
//           segment sizes and of the tile counts;
//   pass 3  every valid route takes slot offs[e] + earlier-chunk count +
//           earlier-round count + rank among equal lanes of its round, which
//           is its rank in ascending flat order: a stable permutation.  Lanes
//           holding the same expert find each other with match_any for short
//           chunks and with one ballot per bit of the expert index for long
//           ones (measured faster at thousands of routes).
// Padding slots get perm = -1 and the tile list (expert, first slot, valid
// rows) is written per expert, several threads per expert when E is small.  Integer work only: results are bit-exact and
// independent of scheduling.
#include <algorithm>

#include "common.cuh"
#include "masked.cuh"

namespace w4a16 {

// Mask of the lanes whose key equals this lane's, for keys below 2^nbits: one
// ballot per key bit (cheaper than match.any when most keys differ).
__device__ __forceinline__ unsigned lanes_with_key(int key, int nbits) {
  unsigned m = 0xFFFFFFFFu;
  for (int b = 0; b < nbits; ++b) {
    const bool bit = (key >> b) & 1;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, bit);
    m &= bit ? bal : ~bal;
  }
  return m;
}

__global__ void __launch_bounds__(kRoutePrepThreads, 1) route_prep_kernel(const RoutePrepParams p) {
  extern __shared__ int32_t sm[];
  const int E = p.E;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  int32_t* hist = sm;                        // [32][E]
  int32_t* cnt = hist + kRoutePrepWarps * E;  // [E]
  int32_t* poff = cnt + E;                   // [E + 1]
  int32_t* toff = poff + E + 1;              // [E + 1]
  int32_t* wsum = toff + E + 1;              // [2][32]

  // The ids come from upstream work and the previous forward may still read
  // this workspace: wait for the preceding grid before touching anything.
  pdl_wait();
  pdl_launch_dependents();

  for (int i = tid; i < kRoutePrepWarps * E; i += kRoutePrepThreads) hist[i] = 0;
  for (int i = tid; i < p.ctr_len; i += kRoutePrepThreads) p.counters[i] = 0;
  if (tid == 0) *p.err = 0;  // the flag reports timeouts since this call
  __syncthreads();

  const int R = p.T * p.k;
  const int chunk = ((R + kRoutePrepWarps - 1) / kRoutePrepWarps + 31) / 32 * 32;
  const int r_begin = warp * chunk;
  const int r_end = min(R, r_begin + chunk);
  const unsigned full = 0xFFFFFFFFu;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int key_bits = 32 - __clz(E);  // keys e + 1 lie in [0, E]
  const bool by_ballot = chunk > 64;    // uniform over the CTA
  auto same_expert = [&](int e) -> unsigned {
    return by_ballot ? lanes_with_key(e + 1, key_bits) : __match_any_sync(full, e);
  };

  auto local_of = [&](int r) -> int {
    if (r >= r_end) return -1;
    const int id = p.ids[r];
    if (id == -1) return -1;
    const long long l = static_cast<long long>(id) - p.expert_offset;
    return (l >= 0 && l < E) ? static_cast<int>(l) : -1;
  };

  // pass 1: per-warp histograms (ids fetched kBatch rounds at a time so the
  // global loads overlap instead of forming a latency chain)
  constexpr int kBatch = 8;
  for (int base = r_begin; base < r_end; base += 32 * kBatch) {
    int eb[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) eb[i] = local_of(base + 32 * i + lane);
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (eb[i] >= 0) atomicAdd(&hist[warp * E + eb[i]], 1);
  }
  __syncthreads();

  // pass 2a: exclusive prefix over warps, per expert; total counts
  for (int e = tid; e < E; e += kRoutePrepThreads) {
    int run = 0;
    for (int w = 0; w < kRoutePrepWarps; ++w) {
      const int t = hist[w * E + e];
      hist[w * E + e] = run;
      run += t;
    }
    cnt[e] = run;
  }
  __syncthreads();

  // pass 2b: exclusive scan over experts (E <= 1024 = one value per thread)
  int v_pad = 0, v_til = 0;
  if (tid < E) {
    const int nt = (cnt[tid] + p.bm - 1) / p.bm;
    v_til = nt;
    v_pad = nt * p.bm;
  }
  const int own_pad = v_pad, own_til = v_til;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(full, v_pad, o);
    const int b = __shfl_up_sync(full, v_til, o);
    if (lane >= o) {
      v_pad += a;
      v_til += b;
    }
  }
  if (lane == 31) {
    wsum[warp] = v_pad;
    wsum[32 + warp] = v_til;
  }
  __syncthreads();
  if (warp == 0) {
    int a = wsum[lane], b = wsum[32 + lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a2 = __shfl_up_sync(full, a, o);
      const int b2 = __shfl_up_sync(full, b, o);
      if (lane >= o) {
        a += a2;
        b += b2;
      }
    }
    wsum[lane] = a;       // inclusive over warps
    wsum[32 + lane] = b;
  }
  __syncthreads();
  if (tid < E) {
    const int pre_pad = (warp > 0 ? wsum[warp - 1] : 0) + v_pad - own_pad;
    const int pre_til = (warp > 0 ? wsum[32 + warp - 1] : 0) + v_til - own_til;
    poff[tid] = pre_pad;
    toff[tid] = pre_til;
    if (tid == E - 1) {
      poff[E] = pre_pad + own_pad;
      toff[E] = pre_til + own_til;
    }
  }
  __syncthreads();

  // pass 3: stable placement
  for (int base = r_begin; base < r_end; base += 32 * kBatch) {
    int eb[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) eb[i] = local_of(base + 32 * i + lane);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int r = base + 32 * i + lane;
      const int e = eb[i];
      const unsigned m = same_expert(e);
      if (e >= 0) {
        const int slot = poff[e] + hist[warp * E + e] + __popc(m & lt_mask);
        p.perm[slot] = r;
        p.inv[r] = slot;
      } else if (r < r_end) {
        p.inv[r] = -1;
      }
      __syncwarp();
      if (e >= 0 && (m & lt_mask) == 0) hist[warp * E + e] += __popc(m);
      __syncwarp();
    }
  }

  // padding slots, tile list, counts and offsets: tpe threads per expert (the
  // largest power of two with E * tpe <= the block), each taking every tpe-th
  // padding slot and tile of its expert
  int tpe = 1;
  while (2 * tpe * E <= kRoutePrepThreads) tpe *= 2;
  for (int i = tid; i < E * tpe; i += kRoutePrepThreads) {
    const int e = i / tpe, sub = i % tpe;
    const int c = cnt[e];
    for (int s = poff[e] + c + sub; s < poff[e + 1]; s += tpe) p.perm[s] = -1;
    const int nt = toff[e + 1] - toff[e];
    for (int t = sub; t < nt; t += tpe) {
      p.tiles[toff[e] + t] = make_int4(e, poff[e] + t * p.bm, min(p.bm, c - t * p.bm), 0);
    }
    if (sub == 0) {
      p.counts[e] = c;
      p.offs[e] = poff[e];
    }
  }
  if (tid == 0) {
    p.offs[E] = poff[E];
    *p.num_tiles = toff[E];
  }
}

// Masked-count layout ("feat(pytorch): add CuTeDSL W4A16 MoE backend"
// (LMDeploy), section Modification: invalid routes and masked expert counts):
// expert-major rows with a count per expert become single routes of weight 1
// (rows past an expert's count: invalid), which route preparation and the
// forward then treat like any other routes.
__global__ void __launch_bounds__(256) masked_routes_kernel(const int32_t* counts, int32_t E, int32_t max_rows,
                                                            int32_t expert_offset, int32_t* ids, float* weights) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t n = static_cast<int64_t>(E) * max_rows;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; r < n; r += stride) {
    const int32_t e = static_cast<int32_t>(r / max_rows);
    const int32_t i = static_cast<int32_t>(r - static_cast<int64_t>(e) * max_rows);
    const int32_t c = min(max(counts[e], 0), max_rows);
    ids[r] = i < c ? expert_offset + e : -1;
    weights[r] = 1.0f;
  }
}

cudaError_t launch_masked_routes(const int32_t* counts, int32_t E, int32_t max_rows, int32_t expert_offset,
                                 int32_t* ids, float* weights, int num_sms, cudaStream_t s, bool pdl) {
  const int64_t n = static_cast<int64_t>(E) * max_rows;
  const int64_t blocks = (n + 255) / 256;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(blocks, 8 * num_sms))));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, masked_routes_kernel, counts, E, max_rows, expert_offset, ids, weights);
}

cudaError_t launch_route_prep(const RoutePrepParams& p, int smem_bytes, cudaStream_t s, bool pdl) {
  // The shared-memory opt-in is a per-device function attribute: set it once
  // for every device this process launches on (more than 48 KB is needed from
  // about 350 experts on).
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool configured_for[64] = {false};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured_for[dev]) {
    e = cudaFuncSetAttribute(route_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    configured_for[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kRoutePrepThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_prep_kernel, p);
}

}  // namespace w4a16
