// Route-layout preparation ("histogram") for the local W4A16 MoE forward.
//
// Follows "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy),
// sections Benchmark (route preparation is part of the timed forward; the
// routes come from a router score / top-k step) and Modification (invalid
// routes and masked expert counts), and "perf: reduce split W4A16 routing and
// output overhead" (FlashInfer), section Description (routing-side
// bookkeeping on the route tiles).
//
// The flat routes r = t*k + j are cut into n_cta contiguous chunks of whole
// tokens, one per CTA, so "earlier CTA" means "smaller flat index".  Two
// kernels (one when a single CTA covers the batch):
//   route_hist_kernel    per-CTA expert counts into cta_hist[c][e]
//                        (shared-memory integer atomics: exact and
//                        order-independent).  Router front end: with logits
//                        given, each warp first takes a token's softmax +
//                        top-k (warp_softmax_topk) and writes its ids and
//                        weights -- the router fused into this pass.
//   route_place_kernel   every CTA sums cta_hist over CTAs (expert totals)
//                        and over the CTAs before it (its base in each
//                        expert's segment), scans the padded segment sizes
//                        and the tile counts over experts, then places its
//                        own routes: 32 warps on contiguous sub-chunks,
//                        per-warp counts, a column prefix over warps, and
//                        within a warp's round of 32 routes the rank among
//                        lanes holding the same expert (match_any for short
//                        sub-chunks, one ballot per key bit for long ones).
//                        A route's slot is its rank in ascending flat order
//                        inside its expert's segment: a stable permutation.
//                        CTA c then writes the padding slots (perm = -1),
//                        tile records (expert, first slot, valid rows) and
//                        counts / offsets of experts e = c, c + n_cta, ...
// Integer work only: results are bit-exact and independent of scheduling.
#include <algorithm>

#include "common.cuh"
#include "masked.cuh"
#include "router.cuh"

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

// Local expert of a global id, -1 for invalid (-1) and other ranks' ids.
__device__ __forceinline__ int local_expert(int32_t id, int32_t expert_offset, int32_t E) {
  if (id == -1) return -1;
  const long long l = static_cast<long long>(id) - expert_offset;
  return (l >= 0 && l < E) ? static_cast<int>(l) : -1;
}

// kPerLane > 0: router front end with kPerLane logits per lane (G <= 32 kPerLane).
template <int kPerLane>
__global__ void __launch_bounds__(kRoutePrepThreads, 1) route_hist_kernel(const RoutePrepParams p) {
  extern __shared__ int32_t sm[];
  int32_t* hist = sm;  // [E]
  const int E = p.E;
  const int tid = threadIdx.x;
  // The ids (or logits) come from upstream work and the previous forward may
  // still read this workspace: wait for the preceding grid first.
  pdl_wait();
  pdl_launch_dependents();
  for (int i = tid; i < E; i += kRoutePrepThreads) hist[i] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * p.tpc;
  const int t1 = min(p.T, t0 + p.tpc);
  if (kPerLane > 0) {
    const int lane = tid & 31;
    for (int t = t0 + (tid >> 5); t < t1; t += kRoutePrepWarps) {
      int32_t* ids = p.ids_out + static_cast<int64_t>(t) * p.k;
      float* wts = p.weights_out + static_cast<int64_t>(t) * p.k;
      warp_softmax_topk<(kPerLane > 0 ? kPerLane : 1)>(p.logits + static_cast<int64_t>(t) * p.G, p.G, p.k, lane,
                                                       [&](int j, int id, float prob) {
                                                         ids[j] = id;
                                                         wts[j] = prob;
                                                         const int e = local_expert(id, p.expert_offset, E);
                                                         if (e >= 0) atomicAdd(&hist[e], 1);
                                                       });
    }
  } else {
    for (int r = t0 * p.k + tid; r < t1 * p.k; r += kRoutePrepThreads) {
      const int e = local_expert(p.ids[r], p.expert_offset, E);
      if (e >= 0) atomicAdd(&hist[e], 1);
    }
  }
  __syncthreads();
  for (int i = tid; i < E; i += kRoutePrepThreads) p.cta_hist[static_cast<int64_t>(blockIdx.x) * E + i] = hist[i];
}

__global__ void __launch_bounds__(kRoutePrepThreads, 1) route_place_kernel(const RoutePrepParams p) {
  extern __shared__ int32_t sm[];
  const int E = p.E;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int cta = blockIdx.x;
  int32_t* whist = sm;                         // [32][E]
  int32_t* cnt = whist + kRoutePrepWarps * E;  // [E] expert totals
  int32_t* cbase = cnt + E;                    // [E] routes of expert e in earlier CTAs
  int32_t* poff = cbase + E;                   // [E + 1]
  int32_t* toff = poff + E + 1;                // [E + 1]
  int32_t* wsum = toff + E + 1;                // [2][32]

  pdl_wait();
  pdl_launch_dependents();

  const int R0 = cta * p.tpc * p.k;
  const int R1 = min(p.T, (cta + 1) * p.tpc) * p.k;
  const int chunk = ((max(R1 - R0, 0) + kRoutePrepWarps - 1) / kRoutePrepWarps + 31) / 32 * 32;
  // warps that hold routes: only their histogram rows are used (small batches
  // touch two or three warps' rows, not 32)
  const int nw = max(1, min(kRoutePrepWarps, (max(R1 - R0, 0) + chunk - 1) / max(chunk, 1)));

  for (int i = tid; i < nw * E; i += kRoutePrepThreads) whist[i] = 0;
  for (int i = cta * kRoutePrepThreads + tid; i < p.ctr_len; i += p.n_cta * kRoutePrepThreads) p.counters[i] = 0;
  if (cta == 0 && tid == 0) *p.err = 0;  // the flag reports timeouts since this call
  __syncthreads();

  const int r_begin = R0 + warp * chunk;
  const int r_end = min(R1, r_begin + chunk);
  const unsigned full = 0xFFFFFFFFu;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int key_bits = 32 - __clz(E);  // keys e + 1 lie in [0, E]
  const bool by_ballot = chunk > 64;    // uniform over the CTA
  auto same_expert = [&](int e) -> unsigned {
    return by_ballot ? lanes_with_key(e + 1, key_bits) : __match_any_sync(full, e);
  };
  auto local_of = [&](int r) -> int { return r < r_end ? local_expert(p.ids[r], p.expert_offset, E) : -1; };

  // pass 1: per-warp counts of this CTA's routes (ids fetched kBatch rounds at
  // a time so the global loads overlap instead of forming a latency chain; a
  // warp with a single batch keeps its experts for pass 3)
  constexpr int kBatch = 8;
  const bool one_batch = chunk <= 32 * kBatch;  // uniform over the CTA
  int eb[kBatch];
  for (int base = r_begin; base < r_end; base += 32 * kBatch) {
#pragma unroll
    for (int i = 0; i < kBatch; ++i) eb[i] = local_of(base + 32 * i + lane);
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (eb[i] >= 0) atomicAdd(&whist[warp * E + eb[i]], 1);
  }
  __syncthreads();

  // pass 2a: exclusive prefix over warps per expert; expert totals and this
  // CTA's base inside each expert's segment (E <= 1024: one expert per thread)
  if (tid < E) {
    const int e = tid;
    int run = 0;
    for (int w = 0; w < nw; ++w) {
      const int t = whist[w * E + e];
      whist[w * E + e] = run;
      run += t;
    }
    if (p.n_cta == 1) {
      cnt[e] = run;
      cbase[e] = 0;
    } else {
      int tot = 0, mine = 0;
      for (int c = 0; c < p.n_cta; ++c) {
        const int v = p.cta_hist[static_cast<int64_t>(c) * E + e];
        mine += c < cta ? v : 0;
        tot += v;
      }
      cnt[e] = tot;
      cbase[e] = mine;
    }
  }
  __syncthreads();

  // pass 2b: exclusive scan over experts of the padded segment sizes and the
  // tile counts
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
    wsum[lane] = a;  // inclusive over warps
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

  // pass 3: stable placement of this CTA's routes
  for (int base = r_begin; base < r_end; base += 32 * kBatch) {
    if (!one_batch) {
#pragma unroll
      for (int i = 0; i < kBatch; ++i) eb[i] = local_of(base + 32 * i + lane);
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int r = base + 32 * i + lane;
      const int e = eb[i];
      const unsigned m = same_expert(e);
      if (e >= 0) {
        const int slot = poff[e] + cbase[e] + whist[warp * E + e] + __popc(m & lt_mask);
        p.perm[slot] = r;
        p.inv[r] = slot;
      } else if (r < r_end) {
        p.inv[r] = -1;
      }
      __syncwarp();
      if (e >= 0 && (m & lt_mask) == 0) whist[warp * E + e] += __popc(m);
      __syncwarp();
    }
  }

  // padding slots, tile list, counts and offsets of this CTA's experts
  // e = cta + i * n_cta: tpe threads per expert (the largest power of two
  // with experts * tpe <= the block), each taking every tpe-th padding slot
  // and tile of its expert
  const int mine_e = cta < E ? (E - cta + p.n_cta - 1) / p.n_cta : 0;  // 0 when n_cta > E and cta >= E
  int tpe = 1;
  if (mine_e > 0)
    while (2 * tpe * mine_e <= kRoutePrepThreads) tpe *= 2;
  for (int i = tid; i < mine_e * tpe; i += kRoutePrepThreads) {
    const int e = cta + (i / tpe) * p.n_cta, sub = i % tpe;
    const int c = cnt[e];
    for (int s = poff[e] + c + sub; s < poff[e + 1]; s += tpe) p.perm[s] = -1;
    const int nt = toff[e + 1] - toff[e];
    for (int t = sub; t < nt; t += tpe) p.tiles[toff[e] + t] = make_int4(e, poff[e] + t * p.bm, min(p.bm, c - t * p.bm), 0);
    if (sub == 0) {
      p.counts[e] = c;
      p.offs[e] = poff[e];
    }
  }
  if (cta == 0 && tid == 0) {
    p.offs[E] = poff[E];
    *p.num_tiles = toff[E];
  }
}

int route_hist_smem(int E) { return E * 4; }
int route_place_smem(int E) { return (kRoutePrepWarps * E + 4 * E + 2 + 64) * 4; }

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

// Masked-count layout written directly by the down GEMM: rows i >= counts[e]
// of every expert are +0 (the GEMM's padding slots may have landed there).
// counts: route preparation's per-expert route counts; 16-bit elements.
__global__ void __launch_bounds__(256) masked_zero_rows_kernel(const int32_t* counts, int32_t max_rows, int32_t H,
                                                               uint4* out) {
  pdl_wait();
  pdl_launch_dependents();
  const int e = blockIdx.y;
  const int c = min(counts[e], max_rows);
  const int vec_row = H / 8;  // 16-byte vectors of a row
  const int64_t n = static_cast<int64_t>(max_rows - c) * vec_row;
  uint4* base = out + (static_cast<int64_t>(e) * max_rows + c) * vec_row;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    base[i] = make_uint4(0u, 0u, 0u, 0u);
}

cudaError_t launch_masked_zero_rows(const int32_t* counts, int32_t E, int32_t max_rows, int32_t H, void* out,
                                    cudaStream_t s, bool pdl) {
  const int64_t per_expert = static_cast<int64_t>(max_rows) * (H / 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>((per_expert + 255) / 256, 64))),
                     static_cast<unsigned>(E));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, masked_zero_rows_kernel, counts, max_rows, H, static_cast<uint4*>(out));
}

namespace {
template <typename K>
cudaError_t launch_rp(K kern, const RoutePrepParams& p, int grid, int smem_bytes, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRoutePrepThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}
}  // namespace

cudaError_t launch_route_prep(const RoutePrepParams& p, cudaStream_t s, bool pdl) {
  // The shared-memory opt-in is a per-device function attribute: set it once
  // for every device this process launches on (route_place_kernel needs more
  // than 48 KB from about 330 experts on).
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool configured_for[64] = {false};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured_for[dev]) {
    e = cudaFuncSetAttribute(route_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, route_place_smem(1024));
    if (e != cudaSuccess) return e;
    configured_for[dev] = true;
  }
  const bool router = p.logits != nullptr;
  if (router || p.n_cta > 1) {
    const int per_lane = (p.G + 31) / 32;
    const int sm_a = route_hist_smem(p.E);
    if (!router) e = launch_rp(route_hist_kernel<0>, p, p.n_cta, sm_a, s, pdl);
    else if (per_lane <= 1) e = launch_rp(route_hist_kernel<1>, p, p.n_cta, sm_a, s, pdl);
    else if (per_lane <= 2) e = launch_rp(route_hist_kernel<2>, p, p.n_cta, sm_a, s, pdl);
    else if (per_lane <= 4) e = launch_rp(route_hist_kernel<4>, p, p.n_cta, sm_a, s, pdl);
    else if (per_lane <= 8) e = launch_rp(route_hist_kernel<8>, p, p.n_cta, sm_a, s, pdl);
    else if (per_lane <= 16) e = launch_rp(route_hist_kernel<16>, p, p.n_cta, sm_a, s, pdl);
    else e = launch_rp(route_hist_kernel<32>, p, p.n_cta, sm_a, s, pdl);
    if (e != cudaSuccess) return e;
  }
  return launch_rp(route_place_kernel, p, p.n_cta, route_place_smem(p.E), s, pdl);
}

}  // namespace w4a16
