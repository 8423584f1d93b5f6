// Expert-grouped W4A16 GEMM for sm_103a (both MoE GEMMs).
//
// Computes, per route tile (expert e, bn consecutive slots) and per 128-row
// weight tile, the swapped product  D[row, route] = sum_k Wq[e][row, k] * B[route, k]
// with the INT4 weights dequantised on chip.  This is the "gate/up GEMM" and
// "down GEMM" of "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy),
// sections Modification (register-side INT4 dequantisation, FP32
// accumulation, TMA buffering, small-batch split-K, route-count-based tile
// selection) and Benchmark; the dequantisation is done by warp-specialised
// warpgroups as in "perf: reduce split W4A16 routing and output overhead"
// (FlashInfer), section Description.  Blackwell design (not the pages'):
//
//   weights (A, M = 128 rows)  TMA (128B swizzle) -> SMEM packed INT4, 256 K
//                              values per stage -> 4 dequant warpgroups, one
//                              64-K quarter of every stage each -> BF16/FP16
//                              A operand in TMEM (a ring of 2 or 3 whole-stage
//                              slots, so dequantisation runs ahead of the MMAs)
//   group scales               TMA boxes of 8 groups (16-byte rows), else cp.async
//   activations (B, N = bn)    gate/up: token rows of x gathered by route with
//                              cp.async (128B-swizzled, K-major; x stays in
//                              L2); down: TMA tiles of the slot-ordered
//                              intermediate
//   tcgen05.mma.kind::f16 (A from TMEM, B from SMEM, N = the tile's valid rows
//   rounded up to 16), FP32 accumulators in TMEM, double-buffered, drained by
//   four epilogue warps; the down GEMM's outputs (activation dtype, or FP32
//   split partials) leave through SMEM staging buffers as TMA tensor stores.
//
// Warp roles (768 threads):
//   warp 0        TMA producer: packed weights, group scales (down GEMM: also
//                 the activation tile)
//   warp 1        TMEM allocation + MMA issuer: the whole warp walks the
//                 pipeline, one elected lane issues (a converged issuer keeps
//                 the tensor pipe fed; a lone lane issued at 2/3 the rate).
//                 One wait and one commit per stage of 16 MMAs: this warp
//                 shares its scheduler with four busy dequant warps, so every
//                 instruction it saves is MMA throughput
//   warps 2, 3    gate/up GEMM: activation-row gather (cp.async); down: idle
//   warps 4..19   four dequant warpgroups; warpgroup h dequantises K-quarter h
//                 of every stage into columns 32 h .. 32 h + 31 of the stage's
//                 TMEM A slot
//   warps 20..23  epilogue (TMEM -> registers -> activation / scaling -> HBM);
//   (24..27)      the down GEMM has a second epilogue set (its epilogue
//                 stores every output element and would otherwise set the
//                 pace); set s takes the unit's weight tiles t with t % 2 == s
// A warp can reach only the TMEM lanes 32 (warp % 4) .. + 31, so dequant and
// epilogue warp w handles weight-tile rows of lane quadrant w % 4.
//
// Work is a persistent loop over units (route tile, group of NT weight tiles,
// K split); every role walks the same unit sequence.  The NT tiles of a unit
// share each stage's activation tile: with one tile per unit the activation
// rows would cross from L2 twice for every byte of weights at 64-route tiles,
// more than the L2-to-SM path carries at the weight-streaming rate.  All waits are bounded (see
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
  __device__ static __forceinline__ float to_float(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
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
  __device__ static __forceinline__ float to_float(uint16_t b) {
    __half h;
    *reinterpret_cast<uint16_t*>(&h) = b;
    return __half2float(h);
  }
};

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Weights packed along K (every layout except per-channel CANON, which packs
// row pairs): 128-row SMEM tile of 2 boxes x 64 rows x 128 bytes.
template <int SCALE, int LAYOUT>
struct KPacked {
  static constexpr bool value = SCALE == SCALE_GROUP || LAYOUT == LAYOUT_IL;
};

// Unit decoding shared by every role: unit u = (route tile, group of NT
// weight tiles, K split), split fastest.
struct Unit {
  int tile, grp, split, kb0, kb1;
  int nsplit;  // K pieces of this unit (1: whole)
  int tj;      // tail pieces: index of the unit among the tail units, else -1
};

__device__ __forceinline__ Unit decode_unit(const GemmParams& p, int u) {
  Unit w;
  w.split = u % p.splits;
  const int r = u / p.splits;
  w.grp = r % p.n_groups;
  w.tile = r / p.n_groups;
  w.kb0 = w.split * p.kb_per_split;
  w.kb1 = min(w.kb0 + p.kb_per_split, p.kb_total);
  w.nsplit = p.splits;
  w.tj = -1;
  return w;
}

// Route-tile record of unit u.  Every unit index below the grid-size bound maps
// to a tile index below the tile-list capacity, so this may be issued before the
// tile count is known (speculatively, to overlap its latency).
__device__ __forceinline__ int4 load_tile(const GemmParams& p, int u) {
  return p.tiles[u / (p.splits * p.n_groups)];
}

// The CTAs take units round robin, so with U units on G CTAs the last wave
// holds U mod G of them and leaves the other SMs idle for a whole unit.  Tail
// pieces (gate/up without split-K only): the first G * floor(U / G) units stay
// whole; each unit of the partial last wave is cut into S K pieces (at most
// tail_max, at most G / (U mod G), every piece owning K blocks), whose partial
// sums the last piece to finish adds up in piece order.
struct UnitMap {
  int main;   // whole units [0, main)
  int S;      // pieces per later unit (1: no tail pieces)
  int kbps;   // K blocks per piece
  int total;  // unit indices
};

template <int WHICH>
__device__ __forceinline__ UnitMap make_unit_map(const GemmParams& p, int n_tiles_rt) {
  const int base = n_tiles_rt * p.n_groups * p.splits;
  UnitMap m{base, 1, p.kb_per_split, base};
  const int G = static_cast<int>(gridDim.x);
  if (WHICH == GEMM_UP && p.splits == 1 && p.tail_max > 1) {
    const int W = base / G, r = base - W * G;
    if (W >= 1 && r > 0) {
      int S = min(min(p.tail_max, p.kb_total), G / r);
      if (S >= 2) {
        const int kbps = (p.kb_total + S - 1) / S;
        S = (p.kb_total + kbps - 1) / kbps;
        m = UnitMap{W * G, S, kbps, W * G + r * S};
      }
    }
  }
  return m;
}

__device__ __forceinline__ Unit decode_unit(const GemmParams& p, const UnitMap& m, int u) {
  if (u < m.main || m.S == 1) return decode_unit(p, u);
  const int v = u - m.main;
  const int b = m.main + v / m.S;  // the whole-unit index (p.splits == 1)
  Unit w;
  w.split = v % m.S;
  w.grp = b % p.n_groups;
  w.tile = b / p.n_groups;
  w.kb0 = w.split * m.kbps;
  w.kb1 = min(w.kb0 + m.kbps, p.kb_total);
  w.nsplit = m.S;
  w.tj = b - m.main;
  return w;
}

__device__ __forceinline__ int4 load_tile(const GemmParams& p, const UnitMap& m, int u) {
  if (u < m.main || m.S == 1) return load_tile(p, u);
  return p.tiles[(m.main + (u - m.main) / m.S) / p.n_groups];
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

// Eight INT4 codes of one 32-bit word -> four 16-bit pairs of consecutive K
// values (k, k + 1), optionally times the scale pair s2.
//   CANON (byte m = K 2m | K 2m+1 << 4): a byte permute moves byte m of the
//   word and of word >> 4 into the two halves first;
//   IL (nibble position p = K {0,2,4,6,1,3,5,7}[p]): shifts alone line the
//   pairs up.
// In both, (v & 0x000F000F) ^ magic is B + q exactly in each half (B = 136 for
// BF16, 1032 for FP16; nibble = q & 15) and subtracting B leaves the exact q.
template <int DT, int LAYOUT, bool SCALED>
__device__ __forceinline__ void codes_of_word(uint32_t x, uint32_t s2, uint32_t* out) {
  using T = F16<DT>;
  const uint32_t kMask = 0x000F000Fu;
  uint32_t p[4];
  if (LAYOUT == LAYOUT_IL) {
    p[0] = x;
    p[1] = x >> 4;
    p[2] = x >> 8;
    p[3] = x >> 12;
  } else {
    const uint32_t sh = x >> 4;
    p[0] = __byte_perm(x, sh, 0x0400);
    p[1] = __byte_perm(x, sh, 0x0501);
    p[2] = __byte_perm(x, sh, 0x0602);
    p[3] = __byte_perm(x, sh, 0x0703);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t q = T::sub(lop3_and_xor(p[i], kMask, T::kMagic), T::kMagic);
    out[i] = SCALED ? T::mul(q, s2) : q;
  }
}

// Dequantise K-quarter h (kQuarterK = 64 K values) of one stage of this
// thread's weight row into TMEM columns [a_col, a_col + 32) of its lane.
//   K-packed layouts: 2 boxes (row block) of 64 rows x 128 B (256 K values)
//   with the 128-byte swizzle (one 16 B chunk = one group of 32); group
//   scales as 128 rows x 16 B (8 groups); the A operand is q * s rounded once
//   to the 16-bit type (group scales) or the exact code q (per-channel: the
//   scale multiplies the FP32 accumulator in the epilogue).
//   per-channel CANON: packed along rows, 4 boxes (row block, K half) of 32
//   row pairs x 128 B with the 128-byte swizzle; the A operand is the exact q.
template <int SCALE, int DT, int LAYOUT>
__device__ __forceinline__ void dequant_quarter(const uint8_t* sA, const uint8_t* sS, int tr, int h,
                                                uint32_t a_taddr) {
  using T = F16<DT>;
  if (KPacked<SCALE, LAYOUT>::value) {
    const uint8_t* row = sA + (tr >> 6) * 8192 + (tr & 63) * 128;
    const int sw = tr & 7;
    uint32_t sword = 0;
    if (SCALE == SCALE_GROUP) sword = *reinterpret_cast<const uint32_t*>(sS + tr * 16 + h * 4);
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const uint4 w = *reinterpret_cast<const uint4*>(row + (((2 * h + g) ^ sw) << 4));
      uint32_t s2 = 0;
      if (SCALE == SCALE_GROUP) {
        const uint16_t s16 = T::from_bf16(static_cast<uint16_t>(sword >> (g * 16)));
        s2 = static_cast<uint32_t>(s16) * 0x00010001u;
      }
      uint32_t out[16];
      codes_of_word<DT, LAYOUT, SCALE == SCALE_GROUP>(w.x, s2, out + 0);
      codes_of_word<DT, LAYOUT, SCALE == SCALE_GROUP>(w.y, s2, out + 4);
      codes_of_word<DT, LAYOUT, SCALE == SCALE_GROUP>(w.z, s2, out + 8);
      codes_of_word<DT, LAYOUT, SCALE == SCALE_GROUP>(w.w, s2, out + 12);
      tmem_st16(a_taddr + 16 * g, out);
    }
  } else {
    const int b = tr >> 6;
    const int lr = tr & 63;
    const int pr = lr >> 1;
    const int shift = (lr & 1) * 4;
    const uint8_t* row = sA + (b * 2 + (h >> 1)) * 4096 + pr * 128;
    const uint32_t kMask = 0x000F000Fu;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const int c = 4 * (h & 1) + cc;  // 16-K chunk of the K half
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
      tmem_st8(a_taddr + cc * 8, out);
    }
  }
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// MMA N for a route tile with `rows` valid routes: rows rounded up to 16
// (kind::f16 with M = 128 takes N in steps of 16), at most bn.
__device__ __forceinline__ int mma_n_of(int rows, int bn) { return min(bn, max(16, (rows + 15) & ~15)); }

// Bounded wait by every lane of a warp, with a warp-uniform result: a lane
// that gave up (timeout or abort) makes the whole warp give up, so no warp is
// left diverged before a __syncwarp or elect.sync.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                          uint64_t limit_ns) {
  const bool r = mbar_wait(bar, parity, abort_flag, err, limit_ns);
  return __all_sync(0xFFFFFFFFu, r);
}

// The MMAs of one A slot (called by the elected lane): NT tiles x 16 / NT
// K16 steps, fully unrolled so that every MMA costs the issuing warp only an
// address add or two -- that warp shares its scheduler with busy dequant
// warps, so its instruction count per MMA bounds the tensor-core rate.
//   d_tmem   accumulator of tile 0 (tile t at + t * bn)
//   a0       the slot's first TMEM column (tile t at + t * 128 / NT)
//   b_j      B descriptor of the slot's first K16 step (64-value atoms of
//            atom_step descriptor units; 32-byte K steps add 2 inside an atom)
//   first    the unit's first slot: each tile's first MMA overwrites
template <int NT>
__device__ __forceinline__ void issue_slot(uint32_t d_tmem, int bn, uint32_t a0, uint64_t b_j, uint32_t atom_step,
                                           uint32_t idesc, bool first, int nvalid) {
  constexpr int kSteps = 16 / NT;  // K16 steps of one tile in a slot
  const uint32_t b_hi = static_cast<uint32_t>(b_j >> 32);
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    if (t < nvalid) {
      const uint32_t d = d_tmem + t * bn;
      uint32_t b_lo = static_cast<uint32_t>(b_j);
#pragma unroll
      for (int kk = 0; kk < kSteps; ++kk) {
        mma_ts_lh(d, a0 + t * (kAslotCols / NT) + kk * 8, b_lo + (kk & 3) * 2, b_hi, idesc,
                  (kk > 0 || !first) ? 1u : 0u);
        if ((kk & 3) == 3) b_lo += atom_step;
      }
    }
  }
}

// MASKED (down GEMM only): the masked-count layout's output [E][max_rows][H]
// takes the expert outputs directly (a separate instance, so that the usual
// one's epilogue code is unchanged).
template <int WHICH, int SCALE, int DT, int LAYOUT, bool MASKED = false>
__global__ void __launch_bounds__(WHICH == GEMM_DOWN ? kGemmThreadsDown : kGemmThreads, 1)
    w4a16_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC,
                      const __grid_constant__ CUtensorMap tmS) {
  using T = F16<DT>;
  constexpr bool kPacked = KPacked<SCALE, LAYOUT>::value;
  constexpr bool kGather = WHICH == GEMM_UP;  // activation rows gathered by cp.async
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived by pointer arithmetic on the shared array so
  // the compiler keeps the shared address space (LDS/STS, not generic loads).
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int stages = p.stages;
  const int bn = p.bn;
  const int NT = p.nt_unit;
  const int acc_bufs = p.acc_bufs;
  const int a_slots = gemm_a_slots(NT, bn, acc_bufs);
  const int acc_col0 = a_slots * kAslotCols;
  // K values of one tile in one A slot (KA = 256 / NT) and 64-K quarters per
  // tile in a slot (qpt = 4 / NT); NT is a power of two
  const int lg_nt = NT == 4 ? 2 : (NT == 2 ? 1 : 0);
  const int qpt = 4 >> lg_nt;
  const int ka_cols = kAslotCols >> lg_nt;  // TMEM columns of one tile in a slot
  // stage layout: NT weight tiles [kStageA each] | activations [bn x 512 B,
  // 4 atoms] | NT scale tiles [kStageS each]
  const int off_b = NT * kStageA;
  const int off_s = off_b + bn * kStageBRow;
  // down GEMM: output staging [8 warps][2][16 x 32] after the stages
  constexpr int kEpiWarps = WHICH == GEMM_DOWN ? 8 : 4;
  float* epi_stage = reinterpret_cast<float*>(smem + stages * p.stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + stages * p.stage_bytes +
                                               (WHICH == GEMM_DOWN ? epi_stage_bytes(p.out16 != 0) : 0));
  uint64_t* empty = full + kMaxStages;
  uint64_t* bfull = empty + kMaxStages;
  uint64_t* afull = bfull + kMaxStages;
  uint64_t* aempty = afull + kMaxAslots;
  uint64_t* accfull = aempty + kMaxAslots;
  uint64_t* accempty = accfull + 2;
  uint64_t* drain = accempty + 2;
  uint64_t* epibar = drain + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(epibar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* fixup_flag = reinterpret_cast<volatile int*>(tmem_holder + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t wait_ns = p.wait_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);                  // producer (TMA bytes + scale copies)
      mbar_init(&empty[s], kGemmDqWarps + 1);  // 16 dequant warps + MMA commit
      mbar_init(&bfull[s], 64);                // the gather warps' 64 lanes
    }
    for (int b = 0; b < a_slots; ++b) {
      mbar_init(&afull[b], kGemmDqWarps);  // every dequant warp (one 64-K quarter each)
      mbar_init(&aempty[b], 1);            // MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], kEpiWarps);
    }
    mbar_init(drain, 1);
    mbar_init(epibar, 4);
    *abort_flag = 0;
    *fixup_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    if (WHICH == GEMM_DOWN) {
      tma_prefetch_desc(&tmB);
      tma_prefetch_desc(&tmC);
    }
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
  // (blockIdx.x < gridDim.x <= the whole units whenever there are tail pieces)
  const int4 first_ti = load_tile(p, blockIdx.x);
  const UnitMap um = make_unit_map<WHICH>(p, *p.num_tiles);
  const int n_units = um.total;
  const int N1 = p.n_rows;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_b = l2_policy_evict_last();
    const bool gated = WHICH == GEMM_UP && p.act == ACT_SWIGLU;
    const bool gate5d = gated && (p.inter % 64) == 0;
    const int groups_row = p.K / kGroup;
    const int sbytes_row = groups_row * 2;
    uint32_t it = 0, ph = 0;
    int st = 0;
    bool ok = true;
    int4 ti_next = first_ti;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit w = decode_unit(p, um, u);
      const int4 ti = ti_next;
      if (u + (int)gridDim.x < n_units) ti_next = load_tile(p, um, u + gridDim.x);  // prefetch
      if (w.kb1 <= w.kb0) continue;
      const int e = ti.x, m0 = ti.y;
      const int nvalid = min(NT, p.n_tiles - w.grp * NT);  // weight tiles of this unit
      const bool scale_copy = SCALE == SCALE_GROUP && !p.scale_tma;
      const uint32_t stage_tx = nvalid * (kStageA + (SCALE == SCALE_GROUP && p.scale_tma ? kStageS : 0)) +
                                (kGather ? 0 : bn * kStageBRow);
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++it, ring_next(st, ph, stages)) {
        if (!warp_wait(&empty[st], ph ^ 1, abort_flag, p.err, wait_ns)) {
          ok = false;
          break;
        }
        uint8_t* sA = smem + st * p.stage_bytes;
        if (scale_copy) {
          // kGroupsPerStage scales (16 B) per tile row; lane handles rows lane + 32 i
          // of every tile; rows beyond the expert's rows read as zero
          const int g0 = kb * kGroupsPerStage;
          const int ng = min(kGroupsPerStage, groups_row - g0);
          for (int t = 0; t < nvalid; ++t) {
            int r0, r1;
            tile_row_bases<WHICH>(p, w.grp * NT + t, r0, r1);
            uint8_t* sS = sA + off_s + t * kStageS;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int tr = lane + 32 * i;
              const int grow = tr < 64 ? r0 + tr : r1 + (tr - 64);
              uint8_t* dst = sS + tr * 16;
              const uint8_t* src = reinterpret_cast<const uint8_t*>(p.scales) +
                                   (static_cast<int64_t>(e) * N1 + grow) * sbytes_row + g0 * 2;
              copy_scale_piece(dst, src, grow < N1 ? max(ng, 0) * 2 : 0);
            }
          }
          cp_async_mbar_arrive(&full[st]);
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[st], stage_tx);
          for (int t = 0; t < nvalid; ++t) {
            int r0, r1;
            tile_row_bases<WHICH>(p, w.grp * NT + t, r0, r1);
            uint8_t* sAt = sA + t * kStageA;
            if (kPacked) {
              // the whole 128-row tile of 128 packed bytes (256 K values) per
              // box, 128-byte swizzle, and its 8 group scales per row: a 5D
              // view pairs a gated tile's 64 gate and 64 up rows, other tiles
              // are 128 consecutive rows (the host encodes the maps by the same
              // rule; gated tiles of an inter that is an odd multiple of 32
              // keep two 64-row boxes)
              uint8_t* sS = sA + off_s + t * kStageS;
              const bool stma = SCALE == SCALE_GROUP && p.scale_tma;
              if (gated && gate5d) {
                tma_load_5d(sAt, &tmA, &full[st], kb * (kBlockK / 2), 0, w.grp * NT + t, 0, e, pol_w);
                if (stma) tma_load_5d(sS, &tmS, &full[st], kb * kGroupsPerStage, 0, w.grp * NT + t, 0, e, pol_w);
              } else if (gated) {
                tma_load_3d(sAt, &tmA, &full[st], kb * (kBlockK / 2), r0, e, pol_w);
                tma_load_3d(sAt + 8192, &tmA, &full[st], kb * (kBlockK / 2), r1, e, pol_w);
                if (stma) {
                  tma_load_3d(sS, &tmS, &full[st], kb * kGroupsPerStage, r0, e, pol_w);
                  tma_load_3d(sS + 1024, &tmS, &full[st], kb * kGroupsPerStage, r1, e, pol_w);
                }
              } else {
                tma_load_3d(sAt, &tmA, &full[st], kb * (kBlockK / 2), r0, e, pol_w);
                if (stma) tma_load_3d(sS, &tmS, &full[st], kb * kGroupsPerStage, r0, e, pol_w);
              }
            } else {
              // four boxes (row block, K half) of 32 row pairs x 128 K bytes, 128-byte swizzle
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                tma_load_3d(sAt + h * 4096, &tmA, &full[st], kb * kBlockK + h * kHalfK, r0 / 2, e, pol_w);
                tma_load_3d(sAt + (2 + h) * 4096, &tmA, &full[st], kb * kBlockK + h * kHalfK, r1 / 2, e, pol_w);
              }
            }
          }
          if (!kGather) {
#pragma unroll
            for (int a = 0; a < kBlockK / 64; ++a)
              tma_load_2d(sA + off_b + a * bn * 128, &tmB, &full[st], kb * kBlockK + a * 64, m0, pol_b);
          }
        }
        __syncwarp();
      }
    }
    // Wind-down: wait (bounded) until the copies of the last stages have
    // landed -- at once after a normal run (the dequantisation warps consumed
    // them), while copies may still be in flight after an abort.
    if (lane == 0) {
      volatile int no_abort = 0;
      for (uint32_t j = (it > (uint32_t)stages ? it - stages : 0); j < it; ++j)
        mbar_wait(&full[j % stages], (j / stages) & 1, &no_abort, p.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp walks the pipeline (every lane waits on the barriers, so
    // the warp stays converged); one elected lane issues.  Per A slot: one
    // wait, 16 MMAs (NT tiles x 256 / NT K values), one commit.
    const uint32_t idesc0 = make_idesc_f16(DT == DT_BF16, kTileRows, 16) & ~(0x3Fu << 17);
    const uint32_t atom_step = static_cast<uint32_t>(bn) * 128 / 16;
    const uint64_t d_stage = static_cast<uint64_t>(p.stage_bytes >> 4);
    const uint64_t bdesc_base = smem_desc_sw128(smem_u32(smem + off_b));
    uint32_t jc = 0, ph = 0, a_ph = 0;
    int st = 0, a_st = 0;
    uint64_t d_st = bdesc_base;  // B descriptor of stage st
    bool ok = true;
    int4 ti_next = first_ti;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit w = decode_unit(p, um, u);
      const int4 ti = ti_next;
      if (u + (int)gridDim.x < n_units) ti_next = load_tile(p, um, u + gridDim.x);
      if (w.kb1 <= w.kb0) continue;
      const uint32_t idesc = idesc0 | (static_cast<uint32_t>(mma_n_of(ti.z, bn) >> 3) << 17);
      const int nvalid = min(NT, p.n_tiles - w.grp * NT);
      const int b = acc_bufs == 2 ? (jc & 1) : 0;
      const uint32_t acc_par = acc_bufs == 2 ? ((jc >> 1) & 1) : (jc & 1);
      if (!warp_wait(&accempty[b], acc_par ^ 1, abort_flag, p.err, wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + acc_col0 + b * NT * bn;
      for (int kb = w.kb0; kb < w.kb1 && ok; ++kb) {
        // gathered activation rows: cp.async writes (generic proxy) become
        // visible to the MMA's shared-memory reads (async proxy) after the
        // barrier and a proxy fence.  The dequant warps arrive on an A slot
        // only after they observed full[st] complete, which also carries the
        // down GEMM's activation bytes, so afull orders both operands there.
        if (kGather) {
          if (!warp_wait(&bfull[st], ph, abort_flag, p.err, wait_ns)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();
        }
        for (int j = 0; j < NT; ++j) {  // the stage's NT A slots, K range j * 256 / NT ..
          if (!warp_wait(&afull[a_st], a_ph, abort_flag, p.err, wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint32_t a0 = tmem + a_st * kAslotCols;
            // slot j covers K16 steps j * 16 / NT .. of the stage: atom j * 4 / NT
            const uint64_t b_j = d_st + static_cast<uint64_t>((j << (2 - lg_nt)) * atom_step);
            const bool first = kb == w.kb0 && j == 0;
            if (NT == 4) issue_slot<4>(d_tmem, bn, a0, b_j, atom_step, idesc, first, nvalid);
            else if (NT == 2) issue_slot<2>(d_tmem, bn, a0, b_j, atom_step, idesc, first, nvalid);
            else issue_slot<1>(d_tmem, bn, a0, b_j, atom_step, idesc, first, nvalid);
            mma_commit(&aempty[a_st]);
          }
          __syncwarp();
          ring_next(a_st, a_ph, a_slots);
        }
        if (!ok) break;
        if (elect_one()) mma_commit(&empty[st]);
        __syncwarp();
        ring_next(st, ph, stages);
        d_st = st == 0 ? bdesc_base : d_st + d_stage;
      }
      if (!ok) break;
      if (elect_one()) mma_commit(&accfull[b]);
      __syncwarp();
      ++jc;
    }
    // Drain: every MMA issued by this warp has finished before TMEM is freed.
    if (elect_one()) mma_commit(drain);
    __syncwarp();
    volatile int no_abort = 0;
    mbar_wait(drain, 0, &no_abort, p.err);
  } else if (warp < 4) {
    // ------------------------------------------------------------------ activation gather
    if (kGather) {
      // Lane l of gather warp g copies 16 bytes (8 K values) of every route row
      // r = g, g + 2, ... of the tile: one row per warp instruction, 512 bytes
      // = this stage's 256 K values, into the 128B-swizzled K-major B tile
      // (atom l / 8, chunk l % 8 of row r at chunk position (l % 8) ^ (r & 7)).
      // Token rows come from x (which stays in L2); K past the end is
      // zero-filled by the copy.  Each lane's cp.async.mbarrier.arrive marks
      // bfull once its copies have landed.
      const int g = warp - 2;
      const uint16_t* xsrc = reinterpret_cast<const uint16_t*>(p.x);
      const int atom = lane >> 3, chunk = lane & 7;
      uint32_t ph = 0;
      int st = 0;
      bool ok = true;
      int4 ti_next = first_ti;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const Unit w = decode_unit(p, um, u);
        const int4 ti = ti_next;
        if (u + (int)gridDim.x < n_units) ti_next = load_tile(p, um, u + gridDim.x);
        if (w.kb1 <= w.kb0) continue;
        const int m0 = ti.y;
        const int rows = min(ti.z, bn);
        // source token of rows g + 2 (lane + 32 i), i < 2 (bn <= 128)
        int src[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = g + 2 * (lane + 32 * i);
          int tok = 0;
          if (r < rows) {
            const int route = p.perm[m0 + r];
            tok = route >= 0 ? route / p.top_k : 0;
          }
          src[i] = tok;
        }
        for (int kb = w.kb0; kb < w.kb1; ++kb, ring_next(st, ph, stages)) {
          if (!warp_wait(&empty[st], ph ^ 1, abort_flag, p.err, wait_ns)) {
            ok = false;
            break;
          }
          uint8_t* sB = smem + st * p.stage_bytes + off_b + atom * bn * 128;
          const int col = kb * kBlockK + lane * 8;
          const bool valid = col < p.K;
          const uint16_t* xcol = xsrc + (valid ? col : 0);
          for (int r = g, i = 0; r < rows; r += 2, ++i) {
            const int tok = __shfl_sync(0xFFFFFFFFu, i < 32 ? src[0] : src[1], i & 31);
            cp_async_cg16(sB + r * 128 + ((chunk ^ (r & 7)) << 4), xcol + static_cast<int64_t>(tok) * p.K,
                          valid ? 16u : 0u);
          }
          cp_async_mbar_arrive_noinc(&bfull[st]);
        }
      }
      // Every copy lands before the CTA exits.
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
  } else if (warp < 4 + kGemmDqWarps) {
    // ------------------------------------------------------------------ dequant warpgroups
    // Warpgroup h fills 64-K quarter h of every A slot: tile h / qpt of the
    // unit, stage quarter j * qpt + h % qpt for the stage's slot j.
    const int h = (warp - 4) >> 2;
    const int q = warp & 3;  // TMEM lane quadrant
    const int tr = tile_row_of_lane<WHICH>(p, q * 32 + lane);
    const int t = h >> (2 - lg_nt);  // h / qpt
    const int hq = h & (qpt - 1);
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16) + t * ka_cols + hq * (kQuarterK / 2);
    uint32_t ph = 0, a_ph = 0;
    int st = 0, a_st = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit w = decode_unit(p, um, u);
      if (w.kb1 <= w.kb0) continue;
      const bool tile_ok = w.grp * NT + t < p.n_tiles;  // uniform over the warpgroup
      for (int kb = w.kb0; kb < w.kb1 && ok; ++kb, ring_next(st, ph, stages)) {
        if (!warp_wait(&full[st], ph, abort_flag, p.err, wait_ns)) {
          ok = false;
          break;
        }
        const uint8_t* sA = smem + st * p.stage_bytes + t * kStageA;
        const uint8_t* sS = smem + st * p.stage_bytes + off_s + t * kStageS;
        for (int j = 0; j < NT; ++j) {
          if (!warp_wait(&aempty[a_st], a_ph ^ 1, abort_flag, p.err, wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (tile_ok) {
            dequant_quarter<SCALE, DT, LAYOUT>(sA, sS, tr, j * qpt + hq, t_lane + a_st * kAslotCols);
            tmem_wait_st();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&afull[a_st]);
          ring_next(a_st, a_ph, a_slots);
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int eset = (warp - (4 + kGemmDqWarps)) >> 2;  // epilogue set: tiles t % 2 == eset (down GEMM)
    const int esets = kEpiWarps / 4;
    const int tr = tile_row_of_lane<WHICH>(p, q * 32 + lane);
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const int epi_tid = threadIdx.x - (4 + kGemmDqWarps) * 32;
    const bool swiglu = (WHICH == GEMM_UP && p.act == ACT_SWIGLU);
    uint32_t jc = 0, eph = 0;
    int sbuf = 0;  // down GEMM: staging buffer of this warp's next chunk
    bool ok = true;
    // Bounded barrier over the four epilogue warps.
    auto epi_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(epibar);
      const bool r = warp_wait(epibar, eph & 1, abort_flag, p.err, wait_ns);
      ++eph;
      return r;
    };
    int4 ti_next = first_ti;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit w = decode_unit(p, um, u);
      const bool has_k = w.kb1 > w.kb0;
      const int4 ti = ti_next;
      if (u + (int)gridDim.x < n_units) ti_next = load_tile(p, um, u + gridDim.x);  // prefetch
      const int e = ti.x, m0 = ti.y, rows = ti.z;
      const int nvalid = min(NT, p.n_tiles - w.grp * NT);
      const int b = acc_bufs == 2 ? (jc & 1) : 0;
      const uint32_t acc_par = acc_bufs == 2 ? ((jc >> 1) & 1) : (jc & 1);
      if (has_k) {
        if (!warp_wait(&accfull[b], acc_par, abort_flag, p.err, wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      for (int t = eset; t < nvalid && ok; t += esets) {
        const int nt = w.grp * NT + t;
        int r0, r1;
        tile_row_bases<WHICH>(p, nt, r0, r1);
        const int grow = tr < 64 ? r0 + tr : r1 + (tr - 64);   // weight row in the expert
        const bool row_ok = swiglu ? (64 * nt + (tr & 63)) < p.inter : grow < N1;
        float scale = 1.0f;
        if (SCALE == SCALE_CHANNEL && row_ok)
          scale = bf16_bits_to_float(p.scales[static_cast<int64_t>(e) * N1 + grow]);
        const uint32_t acc_col = acc_col0 + (b * NT + t) * bn;
        // intermediate column of this lane (SwiGLU: gate/up pair index)
        const int icol = swiglu ? 64 * nt + 16 * q + (lane & 15) : grow;
        // down GEMM: TMEM loads run one 16-route chunk ahead of the conversion
        // and stores (the gate/up epilogue is not on the critical path and
        // keeps its registers for the activation)
        float vn[16];
        if (WHICH == GEMM_DOWN && has_k && rows > 0) tmem_ld16(t_lane + acc_col, vn);
        for (int c0 = 0; c0 < rows; c0 += 16) {
          float v[16];
          if (has_k && WHICH == GEMM_DOWN) {
            tmem_wait_ld(vn);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = vn[j];
            if (c0 + 16 < rows) tmem_ld16(t_lane + acc_col + c0 + 16, vn);
          } else if (has_k) {
            tmem_ld16(t_lane + acc_col + c0, v);
            tmem_wait_ld(v);
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
            // buffers of 16 x 32 output elements: 1 KB (16-bit) or 2 KB (FP32)
            float* stg = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(epi_stage) +
                                                  ((eset * 4 + q) * 2 + sbuf) * (16 * 32 * (p.out16 ? 2 : 4)));
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
              if (MASKED)  // straight into the caller's [E][max_rows][H] output
                tma_store_3d(&tmC, stg, col0, m0 - __ldg(p.seg_offs + e) + c0, e);
              else
                tma_store_2d(&tmC, stg, col0, static_cast<int>(w.split * p.slots_cap) + m0 + c0);
              bulk_commit();
            }
            sbuf ^= 1;
          } else if (w.tj >= 0) {
            // tail piece: [piece][tile][route][TMEM lane], whole rows of 128 lanes
            float* part = p.part + ((static_cast<int64_t>(w.tj) * w.nsplit + w.split) * NT + t) * (p.bn * 128) +
                          q * 32 + lane;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int r = c0 + j;
              if (r < rows) part[r * 128] = v[j];
            }
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
                const float hh = v[j] > 0.0f ? v[j] : 0.0f;
                inter[static_cast<int64_t>(r) * p.inter + icol] = T::from_float(hh * hh);
              }
            }
          }
        }
        if (WHICH == GEMM_UP && w.nsplit > 1) {
          // Split-K fix-up: the last split to finish sums all partials in split
          // order (deterministic) and applies the activation.
          __threadfence();
          if (!epi_sync()) {
            ok = false;
            break;
          }
          if (epi_tid == 0) {
            const int prev = atomicAdd(&p.counters[w.tile * p.n_tiles + nt], 1);
            *fixup_flag = (prev == w.nsplit - 1) ? 1 : 0;
          }
          if (!epi_sync()) {
            ok = false;
            break;
          }
          if (*fixup_flag) {
            __threadfence();
            uint16_t* inter = reinterpret_cast<uint16_t*>(p.out) + static_cast<int64_t>(m0) * p.inter;
            // partials of route r, split s: src + s * sstride + r * rstride
            const float* src;
            int64_t sstride, rstride;
            if (w.tj >= 0) {
              src = p.part + (static_cast<int64_t>(w.tj) * w.nsplit * NT + t) * (p.bn * 128) + q * 32 + lane;
              sstride = static_cast<int64_t>(NT) * p.bn * 128;
              rstride = 128;
            } else {
              src = p.part + static_cast<int64_t>(m0) * N1 + grow;
              sstride = static_cast<int64_t>(p.slots_cap) * N1;
              rstride = N1;
            }
            const bool lane_ok = w.tj >= 0 || row_ok;
            for (int c0 = 0; c0 < rows; c0 += 8) {
              // 8 routes' loads in flight per split, splits summed in order
              float acc[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
              for (int s = 0; s < w.nsplit; ++s) {
                float ld[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  ld[j] = (c0 + j < rows && lane_ok) ? __ldcg(src + s * sstride + (c0 + j) * rstride) : 0.0f;
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] += ld[j];
              }
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int r = c0 + j;
                const float hs = acc[j];
                if (swiglu) {
                  const float other = __shfl_xor_sync(0xFFFFFFFFu, hs, 16);
                  if ((j & 1) == (lane >> 4) && r < rows && row_ok) {
                    const float g = (lane < 16) ? hs : other;
                    const float up = (lane < 16) ? other : hs;
                    inter[static_cast<int64_t>(r) * p.inter + icol] = T::from_float(silu_f(g) * up);
                  }
                } else if (r < rows && row_ok) {
                  const float a = hs > 0.0f ? hs : 0.0f;
                  inter[static_cast<int64_t>(r) * p.inter + icol] = T::from_float(a * a);
                }
              }
            }
            // the flag is rewritten only after the next two barriers
            if (epi_tid == 0) p.counters[w.tile * p.n_tiles + nt] = 0;
          }
        }
      }
      if (!ok) break;
      if (has_k) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&accempty[b]);
        ++jc;
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  if (WHICH == GEMM_DOWN && warp >= 4 + kGemmDqWarps && lane == 0) bulk_wait_all();  // output stores done
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace w4a16

namespace w4a16 {

template <int WHICH, int SCALE, int DT, int LAYOUT, bool MASKED = false>
cudaError_t launch_gemm_one(const GemmParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB,
                            const CUtensorMap& tmC, const CUtensorMap& tmS, int grid, int smem_bytes,
                            cudaStream_t s, bool pdl) {
  auto kern = w4a16_gemm_kernel<WHICH, SCALE, DT, LAYOUT, MASKED>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static int configured_for[64] = {0};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured_for[dev] < smem_bytes) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    configured_for[dev] = smem_bytes;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(WHICH == GEMM_DOWN ? kGemmThreadsDown : kGemmThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, tmA, tmB, tmC, tmS);
}

template <int DT, int LAYOUT>
cudaError_t launch_gemm_dt(int which, int scale_kind, const GemmParams& p, const CUtensorMap& tmA,
                           const CUtensorMap& tmB, const CUtensorMap& tmC, const CUtensorMap& tmS,
                           int grid, int smem_bytes, cudaStream_t s, bool pdl) {
  if (which == GEMM_UP) {
    return scale_kind == SCALE_GROUP
               ? launch_gemm_one<GEMM_UP, SCALE_GROUP, DT, LAYOUT>(p, tmA, tmB, tmC, tmS, grid, smem_bytes, s, pdl)
               : launch_gemm_one<GEMM_UP, SCALE_CHANNEL, DT, LAYOUT>(p, tmA, tmB, tmC, tmS, grid, smem_bytes, s, pdl);
  }
  if (p.masked_rows > 0)
    return scale_kind == SCALE_GROUP
               ? launch_gemm_one<GEMM_DOWN, SCALE_GROUP, DT, LAYOUT, true>(p, tmA, tmB, tmC, tmS, grid, smem_bytes, s,
                                                                             pdl)
               : launch_gemm_one<GEMM_DOWN, SCALE_CHANNEL, DT, LAYOUT, true>(p, tmA, tmB, tmC, tmS, grid, smem_bytes,
                                                                               s, pdl);
  return scale_kind == SCALE_GROUP
             ? launch_gemm_one<GEMM_DOWN, SCALE_GROUP, DT, LAYOUT>(p, tmA, tmB, tmC, tmS, grid, smem_bytes, s, pdl)
             : launch_gemm_one<GEMM_DOWN, SCALE_CHANNEL, DT, LAYOUT>(p, tmA, tmB, tmC, tmS, grid, smem_bytes, s, pdl);
}

}  // namespace w4a16
