// Expert-grouped W4A16 GEMM for sm_103a (both MoE GEMMs).
//
// Computes, per route tile (expert e, bn consecutive slots) and per 128-row
// weight tile, the swapped product  D[row, route] = sum_k Wq[e][row, k] * B[route, k]
// with the INT4 weights dequantised on chip.  This is the "gate/up GEMM" and
// "down GEMM" of "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy),
// sections Modification (register-side INT4 dequantisation, FP32
// accumulation, TMA buffering, small-batch split-K, route-count-based tile
// selection) and Benchmark; the dequantisation is done by two warp-specialised
// warpgroups as in "perf: reduce split W4A16 routing and output overhead"
// (FlashInfer), section Description.  Blackwell design (not the pages'):
//
//   weights (A, M = 128 rows)  TMA (128B swizzle) -> SMEM packed INT4, 256 K
//                              values per stage -> dequant warps -> BF16/FP16
//                              A operand in TMEM (four A buffers of 128 K
//                              values: warpgroup g dequantises K-half g of
//                              every stage into its two buffers, so
//                              dequantisation overlaps the MMAs)
//   group scales               TMA boxes of 8 groups (16-byte rows), else cp.async
//   activations (B, N = bn)    TMA tile of a slot-ordered matrix: the token
//                              rows of x copied by route (gate/up) or the
//                              intermediate (down) -> SMEM (128B-swizzled,
//                              K-major)
//   tcgen05.mma.kind::f16 (A from TMEM, B from SMEM), FP32 accumulators in TMEM,
//   double-buffered, drained by four epilogue warps; the down GEMM's outputs
//   (activation dtype, or FP32 split partials) leave through SMEM staging
//   buffers as TMA tensor stores.
//
// Warp roles (512 threads):
//   warp 0       TMA producer: packed weights, group scales and the activation
//                tile
//   warp 1       TMEM allocation + single-thread MMA issuer
//   warps 2, 3   idle
//   warps 4..11  two dequant warpgroups; warpgroup g dequantises K-half g of
//                every stage into TMEM A buffer (2 * stage counter + g) & 3
//   warps 12..15 epilogue (TMEM -> registers -> activation / scaling -> HBM)
//
// Work is a persistent loop over units (route tile, weight tile, K split);
// every role walks the same unit sequence.  All waits are bounded (see
// mbar_wait): a stuck pipeline raises an error flag and the CTA winds down,
// draining its copies and MMAs before freeing TMEM.
#pragma once
#include "common.cuh"

namespace w4a16 {

// 16-bit type helpers -------------------------------------------------------
template <int DT> struct F16;
template <> struct F16<DT_BF16> {
  // bits of 128 + (nibble ^ 8) in BF16 once ORed/XORed with the nibble, and of 136.0
  static constexpr uint32_t kMagic = 0x43084308u;
  __device__ static __forceinline__ uint32_t sub(uint32_t a, uint32_t b) {
    __nv_bfloat162 r = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&a),
                               *reinterpret_cast<__nv_bfloat162*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
  }
  __device__ static __forceinline__ uint32_t mul(uint32_t a, uint32_t b) {
    __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&a),
                               *reinterpret_cast<__nv_bfloat162*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
  }
  // BF16 scale bits -> this type's bits (identity for BF16)
  __device__ static __forceinline__ uint16_t from_bf16(uint16_t s) { return s; }
  __device__ static __forceinline__ uint16_t from_float(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
  }
};
template <> struct F16<DT_FP16> {
  // FP16: 1024 + (nibble ^ 8) and 1032.0
  static constexpr uint32_t kMagic = 0x64086408u;
  __device__ static __forceinline__ uint32_t sub(uint32_t a, uint32_t b) {
    __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
  }
  __device__ static __forceinline__ uint32_t mul(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
  }
  __device__ static __forceinline__ uint16_t from_bf16(uint16_t s) {
    const float f = __uint_as_float(static_cast<uint32_t>(s) << 16);
    __half h = __float2half_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
  }
  __device__ static __forceinline__ uint16_t from_float(float f) {
    __half h = __float2half_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
  }
};

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Unit decoding shared by every role.
struct Unit {
  int tile, nt, split, kb0, kb1;
};

__device__ __forceinline__ Unit decode_unit(const GemmParams& p, int u) {
  Unit w;
  w.split = u % p.splits;
  const int r = u / p.splits;
  w.nt = r % p.n_tiles;
  w.tile = r / p.n_tiles;
  w.kb0 = w.split * p.kb_per_split;
  w.kb1 = min(w.kb0 + p.kb_per_split, p.kb_total);
  return w;
}

// Route-tile record of unit u.  Every unit index below the grid-size bound maps
// to a tile index below the tile-list capacity, so this may be issued before the
// tile count is known (speculatively, to overlap its latency).
__device__ __forceinline__ int4 load_tile(const GemmParams& p, int u) {
  return p.tiles[u / (p.splits * p.n_tiles)];
}

// Row (within the expert) of the weight rows held in tile rows 0..63 / 64..127.
template <int WHICH>
__device__ __forceinline__ void tile_row_bases(const GemmParams& p, int nt, int& r0, int& r1) {
  if (WHICH == GEMM_UP && p.act == ACT_SWIGLU) {
    r0 = 64 * nt;            // gate rows
    r1 = p.inter + 64 * nt;  // matching up rows
  } else {
    r0 = 128 * nt;
    r1 = 128 * nt + 64;
  }
}

// Tile row (0..127, the row index inside the SMEM weight tile) fed to TMEM lane
// `l`.  For SwiGLU the gate row and the up row of one intermediate index sit in
// lanes l and l ^ 16 of the same warp, so the epilogue pairs them with a shuffle.
template <int WHICH>
__device__ __forceinline__ int tile_row_of_lane(const GemmParams& p, int l) {
  if (WHICH == GEMM_UP && p.act == ACT_SWIGLU) {
    const int q = l >> 5, t = l & 31;
    const int i_local = 16 * q + (t & 15);
    return (t >> 4) ? 64 + i_local : i_local;
  }
  return l;
}

// Dequantise K-half h (kHalfK = 128 K values) of one stage of this thread's
// weight row into TMEM columns [a_col, a_col + 64) of its lane.
//   group scales: 2 boxes (row block) of 64 rows x 128 B (256 K values) with
//   the 128-byte swizzle (one 16 B chunk = one group of 32); scales as 128 rows
//   x 16 B (8 groups); the A operand is q * s rounded once to the 16-bit type.
//   per-channel: packed along rows, 4 boxes (row block, K half) of 32 row pairs
//   x 128 B with the 128-byte swizzle; the A operand is the exact code q (the
//   scale is applied to the FP32 accumulator in the epilogue).
template <int SCALE, int DT>
__device__ __forceinline__ void dequant_stage(const uint8_t* sA, const uint8_t* sS, int tr, int h,
                                              uint32_t a_taddr) {
  using T = F16<DT>;
  const uint32_t kMask = 0x000F000Fu;
  if (SCALE == SCALE_GROUP) {
    const uint2 sc = *reinterpret_cast<const uint2*>(sS + tr * 16 + h * 8);
    const uint8_t* row = sA + (tr >> 6) * 8192 + (tr & 63) * 128;
    const int sw = tr & 7;
    // Compact loop (not unrolled): the body stays small in the instruction
    // cache, which the other warp roles of the CTA share.
#pragma unroll 1
    for (int g = 0; g < kHalfK / kGroup; ++g) {
      const uint4 w = *reinterpret_cast<const uint4*>(row + (((4 * h + g) ^ sw) << 4));
      const uint32_t sword = (g < 2) ? sc.x : sc.y;
      const uint16_t s16 = T::from_bf16(static_cast<uint16_t>(sword >> ((g & 1) * 16)));
      const uint32_t s2 = static_cast<uint32_t>(s16) * 0x00010001u;
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      uint32_t out[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t x = ws[i];
        const uint32_t sh = x >> 4;
        // (k, k+1) = low and high nibble of byte m, moved to the two halves
        const uint32_t p0 = __byte_perm(x, sh, 0x0400);
        const uint32_t p1 = __byte_perm(x, sh, 0x0501);
        const uint32_t p2 = __byte_perm(x, sh, 0x0602);
        const uint32_t p3 = __byte_perm(x, sh, 0x0703);
        out[4 * i + 0] = T::mul(T::sub(lop3_and_xor(p0, kMask, T::kMagic), T::kMagic), s2);
        out[4 * i + 1] = T::mul(T::sub(lop3_and_xor(p1, kMask, T::kMagic), T::kMagic), s2);
        out[4 * i + 2] = T::mul(T::sub(lop3_and_xor(p2, kMask, T::kMagic), T::kMagic), s2);
        out[4 * i + 3] = T::mul(T::sub(lop3_and_xor(p3, kMask, T::kMagic), T::kMagic), s2);
      }
      tmem_st16(a_taddr + 16 * g, out);
    }
  } else {
    const int b = tr >> 6;
    const int lr = tr & 63;
    const int pr = lr >> 1;
    const int shift = (lr & 1) * 4;
    const uint8_t* row = sA + (b * 2 + h) * 4096 + pr * 128;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      const uint4 w = *reinterpret_cast<const uint4*>(row + ((c ^ (pr & 7)) << 4));
      const uint32_t ws[4] = {w.x >> shift, w.y >> shift, w.z >> shift, w.w >> shift};
      uint32_t out[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t p0 = __byte_perm(ws[i], 0, 0x0100);
        const uint32_t p1 = __byte_perm(ws[i], 0, 0x0302);
        out[2 * i + 0] = T::sub(lop3_and_xor(p0, kMask, T::kMagic), T::kMagic);
        out[2 * i + 1] = T::sub(lop3_and_xor(p1, kMask, T::kMagic), T::kMagic);
      }
      tmem_st8(a_taddr + c * 8, out);
    }
  }
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

template <int WHICH, int SCALE, int DT>
__global__ void __launch_bounds__(kGemmThreads, 1)
    w4a16_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC,
                      const __grid_constant__ CUtensorMap tmS) {
  using T = F16<DT>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived by pointer arithmetic on the shared array so
  // the compiler keeps the shared address space (LDS/STS, not generic loads).
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int stages = p.stages;
  const int bn = p.bn;
  // down GEMM: output staging [4 warps][2][16 x 32] after the stages
  float* epi_stage = reinterpret_cast<float*>(smem + stages * p.stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + stages * p.stage_bytes +
                                               (WHICH == GEMM_DOWN ? kEpiStageBytes : 0));
  uint64_t* empty = full + kMaxStages;
  uint64_t* afull = empty + kMaxStages;
  uint64_t* aempty = afull + kNumAbuf;
  uint64_t* accfull = aempty + kNumAbuf;
  uint64_t* accempty = accfull + 2;
  uint64_t* drain = accempty + 2;
  uint64_t* epibar = drain + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(epibar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* fixup_flag = reinterpret_cast<volatile int*>(tmem_holder + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);                  // producer (TMA bytes + scale copies)
      mbar_init(&empty[s], 9);                 // 8 dequant warps + MMA commit
    }
    for (int b = 0; b < kNumAbuf; ++b) {
      mbar_init(&afull[b], 4);
      mbar_init(&aempty[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], 4);
    }
    mbar_init(drain, 1);
    mbar_init(epibar, 4);
    *abort_flag = 0;
    *fixup_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (WHICH == GEMM_DOWN) tma_prefetch_desc(&tmC);
    if (SCALE == SCALE_GROUP && p.scale_tma) tma_prefetch_desc(&tmS);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // Everything below reads what the previous kernels wrote.
  pdl_wait();
  pdl_launch_dependents();

  // The first unit's tile record is fetched together with the tile count.
  const int4 first_ti = load_tile(p, blockIdx.x);
  const int n_units = (*p.num_tiles) * p.n_tiles * p.splits;
  const int N1 = p.n_rows;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_b = l2_policy_evict_last();
    const int groups_row = p.K / kGroup;
    const int sbytes_row = groups_row * 2;
    uint32_t it = 0, ph = 0;
    int st = 0;
    bool ok = true;
    int4 ti_next = first_ti;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit w = decode_unit(p, u);
      const int4 ti = ti_next;
      if (u + (int)gridDim.x < n_units) ti_next = load_tile(p, u + gridDim.x);  // prefetch
      if (w.kb1 <= w.kb0) continue;
      const int e = ti.x, m0 = ti.y;
      int r0, r1;
      tile_row_bases<WHICH>(p, w.nt, r0, r1);
      // cp.async scale rows of this unit for this lane's tile rows (lane + 32 i);
      // null when the row lies beyond the expert's rows
      const bool scale_copy = SCALE == SCALE_GROUP && !p.scale_tma;
      const uint8_t* srow[4];
      bool srow_al16 = true;
      if (scale_copy) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tr = lane + 32 * i;
          const int grow = tr < 64 ? r0 + tr : r1 + (tr - 64);
          srow[i] = grow < N1 ? reinterpret_cast<const uint8_t*>(p.scales) +
                                    (static_cast<int64_t>(e) * N1 + grow) * sbytes_row
                              : nullptr;
          srow_al16 = srow_al16 && ((reinterpret_cast<uintptr_t>(srow[i]) & 15) == 0);
        }
      }
      const uint32_t stage_tx = kStageA + bn * kStageBRow + (SCALE == SCALE_GROUP && p.scale_tma ? kStageS : 0);
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++it, ring_next(st, ph, stages)) {
        if (!mbar_wait(&empty[st], ph ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        uint8_t* sA = smem + st * p.stage_bytes;
        uint8_t* sB = sA + kStageA;
        uint8_t* sS = sB + bn * kStageBRow;
        if (scale_copy) {
          // kGroupsPerStage scales (16 B) per tile row; lane handles rows lane + 32 i.
          const int g0 = kb * kGroupsPerStage;
          const int ng = min(kGroupsPerStage, groups_row - g0);
          if (srow_al16 && ng == kGroupsPerStage) {
            // common case: one 16-byte copy per row
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint8_t* dst = sS + (lane + 32 * i) * 16;
              if (srow[i]) cp_async<16>(dst, srow[i] + g0 * 2);
              else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint8_t* dst = sS + (lane + 32 * i) * 16;
              const int nbytes = srow[i] ? max(ng, 0) * 2 : 0;
              for (int o = 0; o < nbytes; o += 4) cp_async<4>(dst + o, srow[i] + g0 * 2 + o);
              for (int o = nbytes; o < 16; o += 4) *reinterpret_cast<uint32_t*>(dst + o) = 0u;
            }
          }
          cp_async_mbar_arrive(&full[st]);
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[st], stage_tx);
          if (SCALE == SCALE_GROUP) {
            // two 64-row boxes of 128 packed bytes (256 K values), 128-byte swizzle
            tma_load_3d(sA, &tmA, &full[st], kb * (kBlockK / 2), r0, e, pol_w);
            tma_load_3d(sA + 8192, &tmA, &full[st], kb * (kBlockK / 2), r1, e, pol_w);
            if (p.scale_tma) {
              // two 64-row boxes of 8 group scales (16 bytes)
              tma_load_3d(sS, &tmS, &full[st], kb * kGroupsPerStage, r0, e, pol_w);
              tma_load_3d(sS + 1024, &tmS, &full[st], kb * kGroupsPerStage, r1, e, pol_w);
            }
          } else {
            // four boxes (row block, K half) of 32 row pairs x 128 K bytes, 128-byte swizzle
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              tma_load_3d(sA + h * 4096, &tmA, &full[st], kb * kBlockK + h * kHalfK, r0 / 2, e, pol_w);
              tma_load_3d(sA + (2 + h) * 4096, &tmA, &full[st], kb * kBlockK + h * kHalfK, r1 / 2, e,
                          pol_w);
            }
          }
#pragma unroll
          for (int a = 0; a < kBlockK / 64; ++a)
            tma_load_2d(sB + a * bn * 128, &tmB, &full[st], kb * kBlockK + a * 64, m0, pol_b);
        }
        __syncwarp();
      }
    }
    // Wind-down after an abort: wait (bounded) for the copies still in flight.
    if (!ok && lane == 0) {
      volatile int no_abort = 0;
      for (uint32_t j = (it > (uint32_t)stages ? it - stages : 0); j < it; ++j)
        mbar_wait(&full[j % stages], (j / stages) & 1, &no_abort, p.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc_f16(DT == DT_BF16, kTileRows, bn);
      const uint64_t bdesc_base = smem_desc_sw128(smem_u32(smem + kStageA));
      const uint64_t atom_step = static_cast<uint64_t>(bn) * 128 / 16;
      uint32_t it = 0, jc = 0, ph = 0;
      int st = 0;
      uint64_t d_st = bdesc_base;  // B descriptor of stage st
      const uint64_t d_stage = static_cast<uint64_t>(p.stage_bytes >> 4);
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const Unit w = decode_unit(p, u);
        if (w.kb1 <= w.kb0) continue;
        const int b = jc & 1;
        if (!mbar_wait(&accempty[b], ((jc >> 1) & 1) ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + kAccCol0 + b * bn;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          // A: the dequant warps arrive on afull[ab] only after they observed
          // full[st] complete, and full[st] also carries this stage's B bytes
          // (one expect_tx covers weights, scales and activations), so afull
          // alone orders both operands before the MMAs.
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t a_seq = 2 * it + h;
            const int ab = a_seq % kNumAbuf;
            if (!mbar_wait(&afull[ab], (a_seq / kNumAbuf) & 1, abort_flag, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // B descriptors of this stage: the start-address field (bits 0-13,
            // address >> 4) advances by 2 per 32-byte K step inside a 128-byte
            // swizzle atom and by bn * 8 per 64-value atom; adding to the 64-bit
            // value never carries out of the field (shared addresses < 256 KB).
            const uint64_t d0 = d_st + static_cast<uint64_t>(2 * h) * atom_step;
            const uint32_t a0 = tmem + ab * kAbufCols;
            const uint32_t acc0 = (kb > w.kb0 || h > 0) ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < kHalfK / 16; ++kk) {
              mma_ts(d_tmem, a0 + kk * 8, d0 + (kk >> 2) * atom_step + (kk & 3) * 2, idesc,
                     kk > 0 ? 1u : acc0);
            }
            mma_commit(&aempty[ab]);
          }
          if (!ok) break;
          mma_commit(&empty[st]);
          ring_next(st, ph, stages);
          d_st = st == 0 ? bdesc_base : d_st + d_stage;
        }
        if (!ok) break;
        mma_commit(&accfull[b]);
        ++jc;
      }
      // Drain: every MMA issued by this thread has finished before TMEM is freed.
      mma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, p.err);
    }
  } else if (warp < 4) {
    // warps 2 and 3 have no role
  } else if (warp < 12) {
    // ------------------------------------------------------------------ dequant warpgroups
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;
    const int tr = tile_row_of_lane<WHICH>(p, q * 32 + lane);
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t it = 0, ph = 0;
    int st = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit w = decode_unit(p, u);
      if (w.kb1 <= w.kb0) continue;
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++it, ring_next(st, ph, stages)) {
        const uint32_t a_seq = 2 * it + wg;
        const int ab = a_seq % kNumAbuf;
        if (!mbar_wait(&full[st], ph, abort_flag, p.err) ||
            !mbar_wait(&aempty[ab], ((a_seq / kNumAbuf) & 1) ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* sA = smem + st * p.stage_bytes;
        const uint8_t* sS = sA + kStageA + bn * kStageBRow;
        dequant_stage<SCALE, DT>(sA, sS, tr, wg, t_lane + ab * kAbufCols);
        tmem_wait_st();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[ab]);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int tr = tile_row_of_lane<WHICH>(p, q * 32 + lane);
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const int epi_tid = threadIdx.x - 12 * 32;
    const bool swiglu = (WHICH == GEMM_UP && p.act == ACT_SWIGLU);
    uint32_t jc = 0, eph = 0;
    int sbuf = 0;  // down GEMM: staging buffer of this warp's next chunk
    bool ok = true;
    // Bounded barrier over the four epilogue warps.
    auto epi_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(epibar);
      const bool r = mbar_wait(epibar, eph & 1, abort_flag, p.err);
      ++eph;
      return r;
    };
    int4 ti_next = first_ti;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit w = decode_unit(p, u);
      const bool has_k = w.kb1 > w.kb0;
      const int4 ti = ti_next;
      if (u + (int)gridDim.x < n_units) ti_next = load_tile(p, u + gridDim.x);  // prefetch
      const int e = ti.x, m0 = ti.y, rows = ti.z;
      int r0, r1;
      tile_row_bases<WHICH>(p, w.nt, r0, r1);
      const int grow = tr < 64 ? r0 + tr : r1 + (tr - 64);   // weight row in the expert
      const bool row_ok = swiglu ? (64 * w.nt + (tr & 63)) < p.inter : grow < N1;
      float scale = 1.0f;
      if (SCALE == SCALE_CHANNEL && row_ok)
        scale = bf16_bits_to_float(p.scales[static_cast<int64_t>(e) * N1 + grow]);
      const int b = jc & 1;
      if (has_k) {
        if (!mbar_wait(&accfull[b], (jc >> 1) & 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      const uint32_t acc_col = kAccCol0 + b * bn;
      // intermediate column of this lane (SwiGLU: gate/up pair index)
      const int icol = swiglu ? 64 * w.nt + 16 * q + (lane & 15) : grow;
      for (int c0 = 0; c0 < rows; c0 += 16) {
        float v[16];
        if (has_k) {
          tmem_ld16(t_lane + acc_col + c0, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] *= scale;
        if (WHICH == GEMM_DOWN) {
          // This warp's 32 output columns x 16 slots through a staging buffer
          // (slot-major, conflict-free) and one TMA store, in the activation
          // dtype (one rounding) or as FP32 split partials.  Slots past the
          // tile's valid rows are padding slots of y, never read.
          float* stg = epi_stage + (q * 2 + sbuf) * (16 * 32);
          if (lane == 0) bulk_wait_read<1>();  // the store that last read this buffer
          __syncwarp();
          if (p.out16) {
            uint16_t* stg16 = reinterpret_cast<uint16_t*>(stg);
#pragma unroll
            for (int j = 0; j < 16; ++j) stg16[j * 32 + lane] = T::from_float(v[j]);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) stg[j * 32 + lane] = v[j];
          }
          fence_proxy_async_smem();
          __syncwarp();
          const int col0 = grow - lane;
          if (lane == 0 && col0 < p.out_cols) {
            tma_store_2d(&tmC, stg, col0, static_cast<int>(w.split * p.slots_cap) + m0 + c0);
            bulk_commit();
          }
          sbuf ^= 1;
        } else if (p.splits > 1) {
          float* part = p.part + (static_cast<int64_t>(w.split) * p.slots_cap + m0) * N1 + grow;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = c0 + j;
            if (r < rows && row_ok) part[static_cast<int64_t>(r) * N1] = v[j];
          }
        } else {
          uint16_t* inter = reinterpret_cast<uint16_t*>(p.out) + static_cast<int64_t>(m0) * p.inter;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = c0 + j;
            if (swiglu) {
              const float other = __shfl_xor_sync(0xFFFFFFFFu, v[j], 16);
              if ((j & 1) == (lane >> 4) && r < rows && row_ok) {
                const float g = (lane < 16) ? v[j] : other;
                const float up = (lane < 16) ? other : v[j];
                inter[static_cast<int64_t>(r) * p.inter + icol] = T::from_float(silu_f(g) * up);
              }
            } else if (r < rows && row_ok) {
              const float h = v[j] > 0.0f ? v[j] : 0.0f;
              inter[static_cast<int64_t>(r) * p.inter + icol] = T::from_float(h * h);
            }
          }
        }
      }
      if (has_k) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&accempty[b]);
        ++jc;
      }
      if (WHICH == GEMM_UP && p.splits > 1) {
        // Split-K fix-up: the last split to finish sums all partials in split
        // order (deterministic) and applies the activation.
        __threadfence();
        if (!epi_sync()) {
          ok = false;
          break;
        }
        if (epi_tid == 0) {
          const int prev = atomicAdd(&p.counters[w.tile * p.n_tiles + w.nt], 1);
          *fixup_flag = (prev == p.splits - 1) ? 1 : 0;
        }
        if (!epi_sync()) {
          ok = false;
          break;
        }
        if (*fixup_flag) {
          __threadfence();
          uint16_t* inter = reinterpret_cast<uint16_t*>(p.out) + static_cast<int64_t>(m0) * p.inter;
          for (int c0 = 0; c0 < rows; c0 += 16) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int r = c0 + j;
              float h = 0.0f;
              if (r < rows && row_ok) {
                const float* src = p.part + static_cast<int64_t>(m0 + r) * N1 + grow;
                for (int s = 0; s < p.splits; ++s) h += __ldcg(src + static_cast<int64_t>(s) * p.slots_cap * N1);
              }
              if (swiglu) {
                const float other = __shfl_xor_sync(0xFFFFFFFFu, h, 16);
                if ((j & 1) == (lane >> 4) && r < rows && row_ok) {
                  const float g = (lane < 16) ? h : other;
                  const float up = (lane < 16) ? other : h;
                  inter[static_cast<int64_t>(r) * p.inter + icol] = T::from_float(silu_f(g) * up);
                }
              } else if (r < rows && row_ok) {
                const float a = h > 0.0f ? h : 0.0f;
                inter[static_cast<int64_t>(r) * p.inter + icol] = T::from_float(a * a);
              }
            }
          }
          if (epi_tid == 0) p.counters[w.tile * p.n_tiles + w.nt] = 0;
        }
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  if (WHICH == GEMM_DOWN && warp >= 12 && lane == 0) bulk_wait_all();  // output stores done
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace w4a16

namespace w4a16 {

template <int WHICH, int SCALE, int DT>
cudaError_t launch_gemm_one(const GemmParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB,
                            const CUtensorMap& tmC, const CUtensorMap& tmS, int grid, int smem_bytes,
                            cudaStream_t s, bool pdl) {
  auto kern = w4a16_gemm_kernel<WHICH, SCALE, DT>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static int configured_for[64] = {0};
  if (dev < 64 && configured_for[dev] < smem_bytes) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    configured_for[dev] = smem_bytes;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, tmA, tmB, tmC, tmS);
}

template <int DT>
cudaError_t launch_gemm_dt(int which, int scale_kind, const GemmParams& p, const CUtensorMap& tmA,
                           const CUtensorMap& tmB, const CUtensorMap& tmC, const CUtensorMap& tmS,
                           int grid, int smem_bytes, cudaStream_t s, bool pdl) {
  if (which == GEMM_UP) {
    return scale_kind == SCALE_GROUP
               ? launch_gemm_one<GEMM_UP, SCALE_GROUP, DT>(p, tmA, tmB, tmC, tmS, grid, smem_bytes, s, pdl)
               : launch_gemm_one<GEMM_UP, SCALE_CHANNEL, DT>(p, tmA, tmB, tmC, tmS, grid, smem_bytes, s, pdl);
  }
  return scale_kind == SCALE_GROUP
             ? launch_gemm_one<GEMM_DOWN, SCALE_GROUP, DT>(p, tmA, tmB, tmC, tmS, grid, smem_bytes, s, pdl)
             : launch_gemm_one<GEMM_DOWN, SCALE_CHANNEL, DT>(p, tmA, tmB, tmC, tmS, grid, smem_bytes, s, pdl);
}

}  // namespace w4a16
