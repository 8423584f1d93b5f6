// Expert-grouped W4A16 GEMV for sm_103a CUDA cores (both MoE GEMMs, few
// routes per expert).
//
// Same operation, work units and outputs as the tensor-core kernel in gemm.cuh
// (route tile x 128-row weight tile x K split; the "gate/up GEMM" and "down
// GEMM" of "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy), sections
// Modification and Benchmark), for batches where an expert sees only a handful
// of routes.  There each weight is used by 1-4 routes: the contraction is a
// matrix-vector product whose cost is streaming the packed INT4 weights, and a
// tensor-core tile (N >= 16 columns, a fixed issue cost per MMA) would waste
// most of its work.  The route tiles here are at most 16 routes high; each unit
// is run with a compile-time route count R in {1, 2, 3, 4, 8, 16} (the smallest
// that covers the tile).
//
// Arithmetic (per weight row, per 32-element group):
//   * two nibbles of one 32-bit word go to the two FP16 halves with one lop3
//     ((w & mask) ^ magic = FP16 1024 + (nibble ^ 8), or 1024 + 16 (nibble ^ 8)
//     for a nibble in the high half of its byte) and one HSUB2 gives the exact
//     codes q (or 16 q);
//   * the activations are staged in shared memory as FP16, multiplied by a
//     power of two 2^s per (route pair, K block) that puts their largest
//     magnitude in [64, 128) (group scales) or [4, 8) (per-channel scales), and
//     pre-divided by 16 where the weight code is 16 q; so every product q * x
//     is exact and every FP16 partial sum stays below 2^15;
//   * HFMA2 accumulates the 32 products of a group in FP16 (two interleaved
//     chains per route), the group sum is widened to FP32, multiplied by the
//     group scale and accumulated in FP32; 2^-s is applied per K block.
//   Per-channel scales multiply the FP32 total in the epilogue.
//
// Warp roles (320 threads):
//   warp 0     TMA producer of the packed weight tile and the group scales
//              (cp.async), as in the tensor-core kernel
//   warp 1     activation staging: cp.async of the tile's rows (gate/up: token
//              rows of x by slot; down: intermediate rows), then conversion to
//              scaled, permuted FP16 kGemvLag stages later
//   warps 2-9  compute: thread (warp 2 + c, lane l) owns one weight row of the
//              128-row tile and the K half (l >> 4) of every 128-K stage; the
//              halves meet with one shuffle per unit.  For SwiGLU the gate row
//              and the up row of one intermediate index sit in lanes l and
//              l ^ 8 of one warp.
#pragma once
#include "gemm.cuh"

namespace w4a16 {

// Stage layout (bytes from the 1024-aligned stage base).
constexpr int kGvOffS = kStageA;                                // group scales
constexpr int kGvOffRaw = kGvOffS + kStageS;                    // raw activation rows
constexpr int kGvHalfBytes = 144;                               // 64 FP16 + 16 B pad
constexpr int kGvRouteBytes = 2 * kGvHalfBytes;
constexpr int kGvOffX = kGvOffRaw + kGemvMaxR * kStageBRow;     // staged FP16 rows
constexpr int kGvOffInv = kGvOffX + kGemvMaxR * kGvRouteBytes;  // 2^-s per route
static_assert(kGvOffInv + kGemvMaxR * 4 <= kGemvStageBytes, "GEMV stage overflow");
static_assert(kGemvStageBytes % 1024 == 0, "GEMV stages must keep 1024-byte alignment");
constexpr int kGemvLag = 6;  // stages between an activation copy and its conversion
static_assert(kGemvLag + 2 <= kGemvStages, "conversion lag needs a deeper ring");
static_assert(kGemvCtrlBytes >= 3 * kGemvStages * 8 + 8 + 8 + 4 * kGemvStages, "control block");

__device__ __forceinline__ void ring_next(int& st, uint32_t& ph) {
  if (++st == kGemvStages) {
    st = 0;
    ph ^= 1u;
  }
}

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t f2_to_h2_bits(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ __half2 h2_of(uint32_t b) { return *reinterpret_cast<__half2*>(&b); }

// One unit (route tile x weight tile x K split) for a compile-time route count
// R >= rows.  Routes rows..R-1 read stale staging data; their sums are never
// stored.
//
// Codes of one 32-element group, as FP16 pairs matching the staged activations:
//   group scales (K-packed, byte b = K 2b | K 2b+1 << 4): word v holds K
//     8v..8v+7 and gives q[4v..4v+3] = (k0, k4), 16 (k1, k5), (k2, k6), 16 (k3, k7)
//   per-channel (row-pair packed, one byte per K, even row in the low nibble):
//     word j holds K 4j..4j+3 and gives q[2j] = (k0, k2), q[2j + 1] = (k1, k3),
//     times 16 for odd rows
template <int WHICH, int SCALE, int DT, int R>
__device__ __forceinline__ bool gemv_unit(const GemmParams& p, uint8_t* smem, uint64_t* full,
                                          uint64_t* bfull, uint64_t* empty, uint64_t* epibar,
                                          volatile int* abort_flag, volatile int* fixup_flag,
                                          const Unit& w, int e, int m0, int rows, int row,
                                          int cw, int lane, int& st, uint32_t& ph, uint32_t& eph) {
  using T = F16<DT>;
  const int khalf = lane >> 4;
  const bool gated = (WHICH == GEMM_UP && p.act == ACT_SWIGLU);
  const int N1 = p.n_rows;
  float tot[R];
#pragma unroll
  for (int r = 0; r < R; ++r) tot[r] = 0.0f;

  // per-channel: the row's nibble (parity) selects mask and magic
  const uint32_t pc_mask = (row & 1) ? 0x00F000F0u : 0x000F000Fu;
  const uint32_t pc_magic = (row & 1) ? 0x64806480u : 0x64086408u;

  for (int kb = w.kb0; kb < w.kb1; ++kb) {
    if (!mbar_wait(&full[st], ph, abort_flag, p.err) || !mbar_wait(&bfull[st], ph, abort_flag, p.err))
      return false;
    const uint8_t* sA = smem + st * kGemvStageBytes;
    const uint8_t* sX = sA + kGvOffX + khalf * kGvHalfBytes;
    const float* sInv = reinterpret_cast<const float*>(sA + kGvOffInv);
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.0f;
    // this thread's 64 K of packed codes
    uint32_t wd[16];
    uint2 sc = make_uint2(0, 0);
    if (SCALE == SCALE_GROUP) {
      // 64 bytes per row, 64-byte swizzle: 16-byte chunk c sits at c ^ ((row >> 1) & 3)
      const uint8_t* rowp = sA + row * 64;
      const int sw = (row >> 1) & 3;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const uint4 v = *reinterpret_cast<const uint4*>(rowp + (((2 * khalf + g) ^ sw) << 4));
        wd[4 * g + 0] = v.x;
        wd[4 * g + 1] = v.y;
        wd[4 * g + 2] = v.z;
        wd[4 * g + 3] = v.w;
      }
      sc = *reinterpret_cast<const uint2*>(sA + kGvOffS + row * 8);
    } else {
      // two boxes of 32 row pairs x 128 K bytes, 128-byte swizzle
      const int pr = (row & 63) >> 1;
      const uint8_t* rowp = sA + (row >> 6) * 4096 + pr * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(rowp + (((4 * khalf + c) ^ (pr & 7)) << 4));
        wd[4 * c + 0] = v.x;
        wd[4 * c + 1] = v.y;
        wd[4 * c + 2] = v.z;
        wd[4 * c + 3] = v.w;
      }
    }
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      uint32_t q[16];
      if (SCALE == SCALE_GROUP) {
        const uint32_t kLoMask = 0x000F000Fu, kLoMagic = 0x64086408u;  // 1024 + (n ^ 8); 1032
        const uint32_t kHiMask = 0x00F000F0u, kHiMagic = 0x64806480u;  // 1024 + 16 (n ^ 8); 1152
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t wv = wd[4 * g + v];
          const uint32_t w8 = wv >> 8;
          q[4 * v + 0] = hsub2_bits(lop3_and_xor(wv, kLoMask, kLoMagic), kLoMagic);
          q[4 * v + 1] = hsub2_bits(lop3_and_xor(wv, kHiMask, kHiMagic), kHiMagic);
          q[4 * v + 2] = hsub2_bits(lop3_and_xor(w8, kLoMask, kLoMagic), kLoMagic);
          q[4 * v + 3] = hsub2_bits(lop3_and_xor(w8, kHiMask, kHiMagic), kHiMagic);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t wv = wd[8 * g + j];
          q[2 * j + 0] = hsub2_bits(lop3_and_xor(wv, pc_mask, pc_magic), pc_magic);
          q[2 * j + 1] = hsub2_bits(lop3_and_xor(wv >> 8, pc_mask, pc_magic), pc_magic);
        }
      }
      // group scale, BF16 -> FP32 exactly (per-channel: applied in the epilogue)
      float sg = 1.0f;
      if (SCALE == SCALE_GROUP) {
        const int grp = 2 * khalf + g;
        const uint32_t sword = (grp < 2) ? sc.x : sc.y;
        sg = __uint_as_float((grp & 1) ? (sword & 0xFFFF0000u) : (sword << 16));
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint8_t* xr = sX + r * kGvRouteBytes + g * 64;
        __half2 h0 = __float2half2_rn(0.0f), h1 = h0;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xr + v * 16);
          h0 = __hfma2(h2_of(q[4 * v + 0]), h2_of(xv.x), h0);
          h1 = __hfma2(h2_of(q[4 * v + 1]), h2_of(xv.y), h1);
          h0 = __hfma2(h2_of(q[4 * v + 2]), h2_of(xv.z), h0);
          h1 = __hfma2(h2_of(q[4 * v + 3]), h2_of(xv.w), h1);
        }
        const float2 f = __half22float2(__hadd2(h0, h1));
        acc[r] = fmaf(sg, f.x + f.y, acc[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) tot[r] = fmaf(sInv[r], acc[r], tot[r]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    ring_next(st, ph);
  }

  // ---------------------------------------------------------------- epilogue
  // the two K halves of a row: lanes l and l ^ 16
#pragma unroll
  for (int r = 0; r < R; ++r) tot[r] += __shfl_xor_sync(0xFFFFFFFFu, tot[r], 16);
  int r0, r1;
  tile_row_bases<WHICH>(p, w.nt, r0, r1);
  const int grow = row < 64 ? r0 + row : r1 + (row - 64);  // weight row in the expert
  const bool row_ok = gated ? (64 * w.nt + (row & 63)) < p.inter : grow < N1;
  float scale = 1.0f;
  if (SCALE == SCALE_CHANNEL) {
    if (row_ok) scale = bf16_bits_to_float(p.scales[static_cast<int64_t>(e) * N1 + grow]);
    if (row & 1) scale *= 0.0625f;  // odd rows were accumulated as 16 q
  }
  const bool writer = khalf == 0;
  auto epi_sync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(epibar);
    const bool ok = mbar_wait(epibar, eph & 1, abort_flag, p.err);
    ++eph;
    return ok;
  };

  if (WHICH == GEMM_DOWN) {
    float* y = reinterpret_cast<float*>(p.out) +
               (static_cast<int64_t>(w.split) * p.slots_cap + m0) * p.out_cols + grow;
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (writer && r < rows && row_ok) y[static_cast<int64_t>(r) * p.out_cols] = tot[r] * scale;
    return true;
  }

  uint16_t* inter = reinterpret_cast<uint16_t*>(p.out) + static_cast<int64_t>(m0) * p.inter;
  if (p.splits > 1) {
    float* part = p.part + (static_cast<int64_t>(w.split) * p.slots_cap + m0) * N1 + grow;
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (writer && r < rows && row_ok) part[static_cast<int64_t>(r) * N1] = tot[r] * scale;
    // The last split to finish sums the partials in split order
    // (deterministic) and applies the activation.
    __threadfence();
    if (!epi_sync()) return false;
    if (cw == 0 && lane == 0) {
      const int prev = atomicAdd(&p.counters[w.tile * p.n_tiles + w.nt], 1);
      *fixup_flag = (prev == p.splits - 1) ? 1 : 0;
    }
    if (!epi_sync()) return false;
    if (*fixup_flag) {
      __threadfence();
      const int64_t sstride = p.slots_cap * static_cast<int64_t>(N1);
      if (gated) {
        const int i = 64 * w.nt + 8 * cw + lane;
        if (lane < 8 && i < p.inter) {
          for (int r = 0; r < rows; ++r) {
            const float* src = p.part + static_cast<int64_t>(m0 + r) * N1;
            float g = 0.0f, up = 0.0f;
            for (int s = 0; s < p.splits; ++s) {
              g += __ldcg(src + s * sstride + i);
              up += __ldcg(src + s * sstride + p.inter + i);
            }
            inter[static_cast<int64_t>(r) * p.inter + i] = T::from_float(silu_f(g) * up);
          }
        }
      } else if (writer && row_ok) {
        for (int r = 0; r < rows; ++r) {
          const float* src = p.part + static_cast<int64_t>(m0 + r) * N1 + grow;
          float h = 0.0f;
          for (int s = 0; s < p.splits; ++s) h += __ldcg(src + s * sstride);
          const float a = h > 0.0f ? h : 0.0f;
          inter[static_cast<int64_t>(r) * p.inter + grow] = T::from_float(a * a);
        }
      }
      if (cw == 0 && lane == 0) p.counters[w.tile * p.n_tiles + w.nt] = 0;
    }
    return true;
  }

  if (gated) {
    // lanes 0..7: gate rows; lanes 8..15: the matching up rows
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float v = tot[r] * scale;
      const float up = __shfl_xor_sync(0xFFFFFFFFu, v, 8);
      const int i = 64 * w.nt + 8 * cw + (lane & 7);
      if (lane < 8 && r < rows && i < p.inter)
        inter[static_cast<int64_t>(r) * p.inter + i] = T::from_float(silu_f(v) * up);
    }
  } else {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (writer && r < rows && row_ok) {
        const float h = tot[r] * scale;
        const float a = h > 0.0f ? h : 0.0f;
        inter[static_cast<int64_t>(r) * p.inter + grow] = T::from_float(a * a);
      }
    }
  }
  return true;
}

template <int WHICH, int SCALE, int DT>
__global__ void __launch_bounds__(kGemvThreads, 1)
    w4a16_gemv_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmA) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ctrl = smem + kGemvStages * kGemvStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* bfull = full + kGemvStages;
  uint64_t* empty = bfull + kGemvStages;
  uint64_t* epibar = empty + kGemvStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(epibar + 1);
  volatile int* fixup_flag = abort_flag + 1;
  int* stage_rows = reinterpret_cast<int*>(epibar + 2);  // [kGemvStages], staging warp only

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemvStages; ++s) {
      mbar_init(&full[s], 1);    // producer (TMA bytes + scale copies)
      mbar_init(&bfull[s], 1);   // staging warp
      mbar_init(&empty[s], 8);   // compute warps
    }
    mbar_init(epibar, 8);
    *abort_flag = 0;
    *fixup_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tmA);
  __syncthreads();

  // Everything below reads what the previous kernels wrote.
  pdl_wait();
  pdl_launch_dependents();

  const int4 first_ti = load_tile(p, blockIdx.x);
  const int n_units = (*p.num_tiles) * p.n_tiles * p.splits;
  const int N1 = p.n_rows;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    const uint64_t pol_w = l2_policy_evict_first();
    const int groups_row = p.K / kGroup;
    const int sbytes_row = groups_row * 2;
    int st = 0;
    uint32_t ph = 0, issued = 0;
    bool ok = true;
    int4 ti_next = first_ti;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit w = decode_unit(p, u);
      const int4 ti = ti_next;
      if (u + (int)gridDim.x < n_units) ti_next = load_tile(p, u + gridDim.x);
      if (w.kb1 <= w.kb0) continue;
      const int e = ti.x;
      int r0, r1;
      tile_row_bases<WHICH>(p, w.nt, r0, r1);
      const uint8_t* srow[4];
      bool srow_al8 = true;
      if (SCALE == SCALE_GROUP) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tr = lane + 32 * i;
          const int grow = tr < 64 ? r0 + tr : r1 + (tr - 64);
          srow[i] = grow < N1 ? reinterpret_cast<const uint8_t*>(p.scales) +
                                    (static_cast<int64_t>(e) * N1 + grow) * sbytes_row
                              : nullptr;
          srow_al8 = srow_al8 && ((reinterpret_cast<uintptr_t>(srow[i]) & 7) == 0);
        }
      }
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
        if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        uint8_t* sA = smem + st * kGemvStageBytes;
        uint8_t* sS = sA + kGvOffS;
        if (SCALE == SCALE_GROUP) {
          const int g0 = kb * kGroupsPerStage;
          const int ng = min(kGroupsPerStage, groups_row - g0);
          if (srow_al8 && ng == kGroupsPerStage) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint8_t* dst = sS + (lane + 32 * i) * 8;
              if (srow[i]) cp_async<8>(dst, srow[i] + g0 * 2);
              else *reinterpret_cast<uint2*>(dst) = make_uint2(0, 0);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint8_t* dst = sS + (lane + 32 * i) * 8;
              const int nbytes = srow[i] ? max(ng, 0) * 2 : 0;
              for (int o = 0; o < nbytes; o += 4) cp_async<4>(dst + o, srow[i] + g0 * 2 + o);
              for (int o = nbytes; o < 8; o += 4) *reinterpret_cast<uint32_t*>(dst + o) = 0u;
            }
          }
          cp_async_mbar_arrive(&full[st]);
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[st], kStageA);
          if (SCALE == SCALE_GROUP) {
            // two 64-row boxes of 64 packed bytes (128 K values), 64-byte swizzle
            tma_load_3d(sA, &tmA, &full[st], kb * (kBlockK / 2), r0, e, pol_w);
            tma_load_3d(sA + 4096, &tmA, &full[st], kb * (kBlockK / 2), r1, e, pol_w);
          } else {
            // two boxes of 32 row pairs x 128 K bytes, 128-byte swizzle
            tma_load_3d(sA, &tmA, &full[st], kb * kBlockK, r0 / 2, e, pol_w);
            tma_load_3d(sA + 4096, &tmA, &full[st], kb * kBlockK, r1 / 2, e, pol_w);
          }
        }
        __syncwarp();
        ++issued;
        ring_next(st, ph);
      }
    }
    // Wind-down after an abort: wait (bounded) for the copies still in flight.
    if (!ok && lane == 0) {
      volatile int no_abort = 0;
      const uint32_t from = issued > static_cast<uint32_t>(kGemvStages) ? issued - kGemvStages : 0;
      for (uint32_t j = from; j < issued; ++j)
        mbar_wait(&full[j % kGemvStages], (j / kGemvStages) & 1, &no_abort, p.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ activation staging
    // Lanes 0-15 stage route 2i, lanes 16-31 route 2i + 1, 8 K values (16 B)
    // per lane.  Copies land by cp.async; kGemvLag stages later each lane
    // converts what it copied itself (so only its own copies need waiting
    // for), and lane 0 publishes bfull.
    const uint16_t* xsrc = reinterpret_cast<const uint16_t*>(p.x);
    const int hr = lane >> 4, l16 = lane & 15;
    int st = 0, cst = 0;
    uint32_t ph = 0, pending = 0;
    bool ok = true;
    auto convert = [&]() {
      const int rows = stage_rows[cst];
      const uint8_t* raw = smem + cst * kGemvStageBytes + kGvOffRaw;
      uint8_t* xh = smem + cst * kGemvStageBytes + kGvOffX;
      float* inv = reinterpret_cast<float*>(smem + cst * kGemvStageBytes + kGvOffInv);
      for (int rp = 0; rp < rows; rp += 2) {
        const int r = rp + hr;
        float v[8];
        if (r < rows) {
          const uint4 b = *reinterpret_cast<const uint4*>(raw + r * kStageBRow + l16 * 16);
          const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float2 f;
            if (DT == DT_BF16) f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[i]));
            else f = __half22float2(*reinterpret_cast<const __half2*>(&bw[i]));
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = 0.0f;
        }
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
        // largest magnitude of the route pair (the bit patterns of non-negative
        // floats order like the values)
        const uint32_t mb = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m));
        const int ex = static_cast<int>((mb >> 23) & 0xFFu);
        // 2^s puts the maximum in [2^6, 2^7) (group) or [2^2, 2^3) (per-channel)
        int s = (ex == 0 || ex == 255) ? 0 : ((SCALE == SCALE_GROUP ? 133 : 129) - ex);
        s = max(-100, min(100, s));
        const float sc = __uint_as_float(static_cast<uint32_t>(s + 127) << 23);
        uint4 o;
        if (SCALE == SCALE_GROUP) {
          // (x0, x4), (x1, x5) / 16, (x2, x6), (x3, x7) / 16
          const float sc16 = sc * 0.0625f;
          o.x = f2_to_h2_bits(v[0] * sc, v[4] * sc);
          o.y = f2_to_h2_bits(v[1] * sc16, v[5] * sc16);
          o.z = f2_to_h2_bits(v[2] * sc, v[6] * sc);
          o.w = f2_to_h2_bits(v[3] * sc16, v[7] * sc16);
        } else {
          // (x0, x2), (x1, x3), (x4, x6), (x5, x7)
          o.x = f2_to_h2_bits(v[0] * sc, v[2] * sc);
          o.y = f2_to_h2_bits(v[1] * sc, v[3] * sc);
          o.z = f2_to_h2_bits(v[4] * sc, v[6] * sc);
          o.w = f2_to_h2_bits(v[5] * sc, v[7] * sc);
        }
        if (r < rows) {
          *reinterpret_cast<uint4*>(xh + r * kGvRouteBytes + (l16 >> 3) * kGvHalfBytes + (l16 & 7) * 16) = o;
          if (l16 == 0) inv[r] = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bfull[cst]);
      if (++cst == kGemvStages) cst = 0;
      --pending;
    };
    int4 ti_next = first_ti;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit w = decode_unit(p, u);
      const int4 ti = ti_next;
      if (u + (int)gridDim.x < n_units) ti_next = load_tile(p, u + gridDim.x);
      if (w.kb1 <= w.kb0) continue;
      const int m0 = ti.y, rows = min(ti.z, kGemvMaxR);
      // source row of route `lane` (lanes below rows)
      int src = 0;
      if (lane < rows) {
        if (WHICH == GEMM_UP) {
          const int route = p.perm[m0 + lane];
          src = route >= 0 ? route / p.top_k : 0;
        } else {
          src = m0 + lane;
        }
      }
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
        if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        if (lane == 0) stage_rows[st] = rows;
        uint8_t* raw = smem + st * kGemvStageBytes + kGvOffRaw;
        const int col = kb * kBlockK + l16 * 8;
        const bool valid = col < p.K;
        for (int rp = 0; rp < rows; rp += 2) {
          const int r = rp + hr;
          const int srow = __shfl_sync(0xFFFFFFFFu, src, r & 31);
          if (r < rows)
            cp_async_cg16(raw + r * kStageBRow + l16 * 16,
                          xsrc + static_cast<int64_t>(srow) * p.K + (valid ? col : 0), valid ? 16u : 0u);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        __syncwarp();
        ++pending;
        ring_next(st, ph);
        if (pending > static_cast<uint32_t>(kGemvLag)) {
          asm volatile("cp.async.wait_group %0;" ::"n"(kGemvLag) : "memory");
          __syncwarp();
          convert();
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
    while (ok && pending > 0) convert();
  } else {
    // ------------------------------------------------------------------ compute + epilogue
    const int cw = warp - 2;
    const int l16 = lane & 15;
    const bool gated = (WHICH == GEMM_UP && p.act == ACT_SWIGLU);
    const int row = gated ? ((l16 >> 3) * 64 + 8 * cw + (l16 & 7)) : (16 * cw + l16);
    int st = 0;
    uint32_t ph = 0, eph = 0;
    int4 ti_next = first_ti;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const Unit w = decode_unit(p, u);
      const int4 ti = ti_next;
      if (u + (int)gridDim.x < n_units) ti_next = load_tile(p, u + gridDim.x);
      const int e = ti.x, m0 = ti.y, rows = min(ti.z, kGemvMaxR);
      bool ok;
#define W4A16_GEMV_UNIT(RR)                                                                     \
  gemv_unit<WHICH, SCALE, DT, RR>(p, smem, full, bfull, empty, epibar, abort_flag, fixup_flag, \
                                  w, e, m0, rows, row, cw, lane, st, ph, eph)
      if (rows <= 1) ok = W4A16_GEMV_UNIT(1);
      else if (rows <= 2) ok = W4A16_GEMV_UNIT(2);
      else if (rows <= 3) ok = W4A16_GEMV_UNIT(3);
      else if (rows <= 4) ok = W4A16_GEMV_UNIT(4);
      else if (rows <= 8) ok = W4A16_GEMV_UNIT(8);
      else ok = W4A16_GEMV_UNIT(16);
#undef W4A16_GEMV_UNIT
      if (!ok) break;
    }
  }
  __syncthreads();
}

template <int WHICH, int SCALE, int DT>
cudaError_t launch_gemv_one(const GemmParams& p, const CUtensorMap& tmA, int grid, cudaStream_t s,
                            bool pdl) {
  auto kern = w4a16_gemv_kernel<WHICH, SCALE, DT>;
  const int smem_bytes = gemv_smem_bytes();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool configured_for[64] = {false};
  if (dev < 64 && !configured_for[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    configured_for[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, tmA);
}

template <int DT>
cudaError_t launch_gemv_dt(int which, int scale_kind, const GemmParams& p, const CUtensorMap& tmA,
                           int grid, cudaStream_t s, bool pdl) {
  if (which == GEMM_UP) {
    return scale_kind == SCALE_GROUP ? launch_gemv_one<GEMM_UP, SCALE_GROUP, DT>(p, tmA, grid, s, pdl)
                                     : launch_gemv_one<GEMM_UP, SCALE_CHANNEL, DT>(p, tmA, grid, s, pdl);
  }
  return scale_kind == SCALE_GROUP ? launch_gemv_one<GEMM_DOWN, SCALE_GROUP, DT>(p, tmA, grid, s, pdl)
                                   : launch_gemv_one<GEMM_DOWN, SCALE_CHANNEL, DT>(p, tmA, grid, s, pdl);
}

}  // namespace w4a16
