// Expert-grouped W4A16 GEMV for sm_103a (both MoE GEMMs, up to ~12 routes per
// expert), on warp-level MMAs fed by register-side dequantisation.
//
// Same operation, work units and outputs as the tcgen05 kernel in gemm.cuh
// (route tile x 128-row weight tile x K split; the "gate/up GEMM" and "down
// GEMM" of "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy), sections
// Modification and Benchmark), for batches where an expert sees only a few
// routes.  There each weight is used by a handful of routes: the contraction
// is a thin product whose cost is streaming the packed INT4 weights, and a
// 128-row tcgen05 tile with TMEM staging has a fixed cost per MMA that such
// thin tiles cannot amortise.  Here a route tile (<= kGemvMaxR = 32 routes) is
// the N side of mma.sync m16n8k16 -- up to four N = 8 blocks sharing each
// dequantised A fragment -- and the dequantised weights go to the MMAs
// straight from registers.
//
// Arithmetic (per weight row, per 32-element group), in the activation type
// (BF16 or FP16) with FP32 accumulation:
//   * a nibble goes to each 16-bit half of a register with one lop3
//     ((w & 0x000F000F) ^ magic = B + q exactly, B = 136 for BF16 and 1032
//     for FP16, nibble = q & 15) and one HSUB2 of B leaves the exact code q;
//     shifting the word by 4, 8 and 12 bits gives the other three nibble pairs;
//   * the MMA multiplies the exact codes by the activations as given and sums
//     in FP32, one group (two MMAs per N block) at a time; the group result is
//     multiplied by the group scale and accumulated in FP32.
//   Per-channel scales multiply the FP32 total in the epilogue.
//
// A pipeline stage is 128 weight rows x kGemvBlockK (256) K values: 128 bytes
// of every packed row per visit, read by TMA in 128-byte-swizzled boxes.
// With the relaid-out weights (LAYOUT_IL, see common.cuh) every layout is
// packed along K and each code pair holds consecutive K values, so the
// activations feed the MMAs as stored (no byte permutes); per-channel weights
// then take the group-scale data path without the group scales.
//
// Compute mapping: 16 warps = 8 row blocks (16 rows each) x 2 groups.
//   * units of several stages: group h takes K half h of every stage; the
//     halves meet once per unit through a double-buffered shared exchange;
//   * single-stage units without split (e.g. the down GEMM at I = 256): group
//     h takes the units of ordinal parity h over the full K, no exchange.
// In the second case each group has a ring of stages of its own (see
// gemv_unit for why every consumer of a ring sees every phase of it).
//
// Warp roles (576 threads):
//   warp 0      TMA producer of the packed weight tile and the group scales
//               (TMA when their rows are 16-byte multiples, else cp.async)
//   warp 1      activation rows: cp.async of the tile's rows (gate/up: token
//               rows of x by slot; down: intermediate rows), completion
//               signalled on the stage's mbarrier without blocking the warp
//   One mbarrier per stage completes on the producer's TMA bytes and arrival
//   plus one cp.async-tracked arrival per lane of warp 1, so the compute warps
//   wait once per stage (two waits per stage cost ~7 % at 8 to 256 tokens:
//   every poll takes issue slots from the dequantisation).  After an abort
//   warp 1 completes, without copying, the arrivals it owes to stages the
//   producer issued, so that the producer can drain its copies.
//   warps 2-17  compute: warp 2 + c is in group c / 8 and takes row block
//               c % 8 (16 rows: MMA rows g and g + 8).  For SwiGLU a row block
//               holds 8 gate rows and their 8 up rows, so the activation is
//               applied in registers.
#pragma once
#include "gemm.cuh"

namespace w4a16 {

// Stage layout (bytes from the 1024-aligned stage base); the activation rows
// take the rest of the stage (gemv_stage_bytes).
constexpr int kGvWeightBytes = kTileRows * kGemvBlockK / 2;          // packed weights
constexpr int kGvScaleRowBytes = kGemvBlockK / kGroup * 2;            // 8 BF16 scales per row
constexpr int kGvOffS = kGvWeightBytes;
constexpr int kGvOffX = kGvOffS + kTileRows * kGvScaleRowBytes;       // activation rows
constexpr int kGvRouteBytes = kGemvBlockK * 2 + 64;                   // + pad: 64 mod 128
static_assert(kGvRouteBytes == 576, "stage size formula");
constexpr int kGemvMaxNB = kGemvMaxR / 8;
constexpr int kGemvComputeWarps = 16;
static_assert(kGemvThreads == 32 * (2 + kGemvComputeWarps), "warp roles");
// Arrivals that complete a stage: the producer's expect-tx arrival and one
// cp.async-tracked arrival per lane of the activation warp.
constexpr int kGvFullArrivals = 1 + 32;
// Control block: mbarriers and flags, then the tile records of the CTA's first
// kGemvTileTab units from kGvCtrlTabOff, then (units of several stages) the
// K-half exchange from kGvCtrlRedOff: two buffers of 8 warps x NB blocks x 32
// lanes x 4 floats (gemv_ctrl_bytes).
constexpr int kGvCtrlTabOff = 512;
constexpr int kGvCtrlRedOff = kGemvCtrlBytes;
constexpr int kGemvTileTab = 256;
// mbarriers full / empty, the group barrier, abort and fix-up flags, the
// producer's stage counts per ring and its stop flag
static_assert(2 * kGemvMaxStages * 8 + 8 + 8 + 12 <= kGvCtrlTabOff, "control block");
static_assert(kGvCtrlTabOff + kGemvTileTab * 16 <= kGemvCtrlBytes, "tile table");
static_assert(kGemvTileTab <= kGemvThreads, "one record per thread");
static_assert(gemv_smem_bytes(kGemvMaxR, true) <= kGemvSmemLimit && gemv_stages(kGemvMaxR, true) >= 4, "smem");

// Tile record of this CTA's i-th unit u: from the shared table (filled at
// kernel start) or, past its end, from global memory.
__device__ __forceinline__ int4 tile_of(const GemmParams& p, const int4* tab, int i, int u) {
  return i < kGemvTileTab ? tab[i] : load_tile(p, u);
}

// One unit of the CUDA-core path: (route tile, 128-row weight tile nt, K split).
struct GvUnit {
  int tile, nt, split, kb0, kb1;
};

// Iterates this CTA's units u = blockIdx.x + i * gridDim.x, keeping the
// (split, weight tile, route tile) digits of u up to date with carries instead
// of divisions.
struct UnitIter {
  int u, split, nt, tile, ds, dnt, dtile;
  __device__ __forceinline__ void init(const GemmParams& p) {
    u = blockIdx.x;
    split = u % p.splits;
    const int r = u / p.splits;
    nt = r % p.n_tiles;
    tile = r / p.n_tiles;
    const int G = gridDim.x;
    ds = G % p.splits;
    const int gr = G / p.splits;
    dnt = gr % p.n_tiles;
    dtile = gr / p.n_tiles;
  }
  __device__ __forceinline__ void next(const GemmParams& p) {
    u += gridDim.x;
    split += ds;
    int c = 0;
    if (split >= p.splits) {
      split -= p.splits;
      c = 1;
    }
    nt += dnt + c;
    c = 0;
    if (nt >= p.n_tiles) {
      nt -= p.n_tiles;
      c = 1;
    }
    tile += dtile + c;
  }
  __device__ __forceinline__ GvUnit unit(const GemmParams& p) const {
    GvUnit w;
    w.split = split;
    w.nt = nt;
    w.tile = tile;
    w.kb0 = split * p.kb_per_split;
    w.kb1 = min(w.kb0 + p.kb_per_split, p.kb_total);
    return w;
  }
};

// D (16 x 8, FP32) += A (16 x 16) * B (16 x 8), A and B in the activation
// type; fragments as the PTX ISA gives them for m16n8k16: lane (g = lane / 4,
// t = lane % 4) holds A rows g and g + 8 at K 2t, 2t + 1 (a0, a1) and 2t + 8,
// 2t + 9 (a2, a3), B column g at the same K (b0, b1), D rows g, g + 8 at
// columns 2t, 2t + 1.
template <int DT>
__device__ __forceinline__ void mma_16816(float& d0, float& d1, float& d2, float& d3, uint32_t a0, uint32_t a1,
                                          uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  if (DT == DT_BF16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Exact code pair q of the low nibbles of the two 16-bit halves of v:
// (v & 0x000F000F) ^ magic = B + q exactly (B = 136 for BF16, 1032 for FP16;
// nibble = q & 15), minus B.
template <int DT>
__device__ __forceinline__ uint32_t code_pair(uint32_t v) {
  return F16<DT>::sub(lop3_and_xor(v, 0x000F000Fu, F16<DT>::kMagic), F16<DT>::kMagic);
}

// Four 8 x 8 b16 matrices from shared memory; lane l gives the address of row
// l % 8 of matrix l / 8 and receives bytes 4 (l % 4) .. + 3 of row l / 4 of
// each matrix.
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// One stage of one compute warp: 16 weight rows (MMA rows g: rowA, g + 8:
// rowB) x the full stage K (FULLK) or its half kh x NB blocks of 8 routes (MMA columns; columns past
// the route count read stale data and are never stored).  tot[4 n + 0..1]:
// rowA x routes 8 n + 2t, + 1; tot[4 n + 2..3]: rowB x the same routes.
//
// K order inside an MMA: any bijection works as long as A and B agree, so each
// lane feeds whole packed words in the order the nibble extraction yields and
// pairs its activations the same way with byte permutes:
//   group scales (K-packed, byte b = K 2b | K 2b+1 << 4): lane t takes word t
//     of group c's 16-byte chunk (K 32c + 8t .. + 7; one ldmatrix.x4 fetches
//     it for rowA and rowB and two groups); its code pairs (k0, k4), (k1, k5),
//     (k2, k6), (k3, k7) feed MMAs whose sum over the four lanes is exactly
//     group c, so the group scale multiplies that result;
//   per-channel (row-pair packed, one byte per K, even row in the low nibble):
//     lane t takes 16-byte chunks t and t + 4 of each K half; word i of a chunk
//     (4 K) gives (k0, k2) and (k1, k3) for one MMA.
template <int SCALE, int DT, int LAYOUT, int NB, bool FULLK>
__device__ __forceinline__ void gemv_stage(const uint8_t* sA, int rowA, int rowB, int kh, int lane,
                                           uint32_t ld_row_off, int ld_row7, int ld_chunk, float (&tot)[4 * NB]) {
  const int g = lane >> 2, t = lane & 3;
  const uint8_t* sX = sA + kGvOffX + g * kGvRouteBytes;  // this lane's B column in block 0 (route g)
  if (SCALE == SCALE_GROUP || LAYOUT == LAYOUT_IL) {
    constexpr bool kScaled = SCALE == SCALE_GROUP;
    // BF16 scales of the groups this warp handles, two per word: word pp holds
    // the groups of ldmatrix step pp
    uint32_t saw[4] = {0u, 0u, 0u, 0u}, sbw[4] = {0u, 0u, 0u, 0u};
    if (!kScaled) {
    } else if (FULLK) {
      const uint4 sa = *reinterpret_cast<const uint4*>(sA + kGvOffS + rowA * kGvScaleRowBytes);
      const uint4 sb = *reinterpret_cast<const uint4*>(sA + kGvOffS + rowB * kGvScaleRowBytes);
      saw[0] = sa.x; saw[1] = sa.y; saw[2] = sa.z; saw[3] = sa.w;
      sbw[0] = sb.x; sbw[1] = sb.y; sbw[2] = sb.z; sbw[3] = sb.w;
    } else {
      const uint2 sa = *reinterpret_cast<const uint2*>(sA + kGvOffS + rowA * kGvScaleRowBytes + kh * 8);
      const uint2 sb = *reinterpret_cast<const uint2*>(sA + kGvOffS + rowB * kGvScaleRowBytes + kh * 8);
      saw[0] = sa.x; saw[1] = sa.y; saw[2] = 0u; saw[3] = 0u;
      sbw[0] = sb.x; sbw[1] = sb.y; sbw[2] = 0u; sbw[3] = 0u;
    }
    const uint32_t sbase = smem_u32(sA);
#pragma unroll
    for (int pp = 0; pp < (FULLK ? 4 : 2); ++pp) {
      const int pq = FULLK ? pp : 2 * kh + pp;
      // words t of rowA / rowB in groups 2 pq and 2 pq + 1 (128-byte swizzle:
      // chunk c of row r at c ^ (r & 7))
      uint32_t w4[4];
      ldmatrix_x4(sbase + ld_row_off + (((2 * pq + ld_chunk) ^ ld_row7) << 4), w4[0], w4[1], w4[2], w4[3]);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int c = 2 * pq + q;  // group of the stage
        const uint32_t wa = w4[2 * q], wb = w4[2 * q + 1];
        const uint32_t a0 = code_pair<DT>(wa), a1 = code_pair<DT>(wb);
        const uint32_t a2 = code_pair<DT>(wa >> 4), a3 = code_pair<DT>(wb >> 4);
        const uint32_t a4 = code_pair<DT>(wa >> 8), a5 = code_pair<DT>(wb >> 8);
        const uint32_t a6 = code_pair<DT>(wa >> 12), a7 = code_pair<DT>(wb >> 12);
        // BF16 group scales of rowA / rowB -> FP32 exactly
        const float fa = __uint_as_float(q ? (saw[pp] & 0xFFFF0000u) : (saw[pp] << 16));
        const float fb = __uint_as_float(q ? (sbw[pp] & 0xFFFF0000u) : (sbw[pp] << 16));
#pragma unroll
        for (int n = 0; n < NB; ++n) {
          // activations K 32c + 8t .. + 7 of route 8n + g: (x0 x1) (x2 x3) (x4 x5) (x6 x7)
          const uint4 xv = *reinterpret_cast<const uint4*>(sX + n * 8 * kGvRouteBytes + (4 * c + t) * 16);
          // B pairs in the codes' K order: CANON codes pair (k0 k4) (k1 k5) | (k2 k6) (k3 k7),
          // IL codes pair (k0 k1) (k2 k3) | (k4 k5) (k6 k7), i.e. the words as stored
          const uint32_t b0 = LAYOUT == LAYOUT_IL ? xv.x : __byte_perm(xv.x, xv.z, 0x5410);
          const uint32_t b1 = LAYOUT == LAYOUT_IL ? xv.y : __byte_perm(xv.x, xv.z, 0x7632);
          const uint32_t b2 = LAYOUT == LAYOUT_IL ? xv.z : __byte_perm(xv.y, xv.w, 0x5410);
          const uint32_t b3 = LAYOUT == LAYOUT_IL ? xv.w : __byte_perm(xv.y, xv.w, 0x7632);
          if (kScaled) {
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            mma_16816<DT>(d[0], d[1], d[2], d[3], a0, a1, a2, a3, b0, b1);
            mma_16816<DT>(d[0], d[1], d[2], d[3], a4, a5, a6, a7, b2, b3);
            tot[4 * n + 0] = fmaf(fa, d[0], tot[4 * n + 0]);
            tot[4 * n + 1] = fmaf(fa, d[1], tot[4 * n + 1]);
            tot[4 * n + 2] = fmaf(fb, d[2], tot[4 * n + 2]);
            tot[4 * n + 3] = fmaf(fb, d[3], tot[4 * n + 3]);
          } else {
            // exact codes: the per-channel scale multiplies the total in the epilogue
            mma_16816<DT>(tot[4 * n + 0], tot[4 * n + 1], tot[4 * n + 2], tot[4 * n + 3], a0, a1, a2, a3, b0, b1);
            mma_16816<DT>(tot[4 * n + 0], tot[4 * n + 1], tot[4 * n + 2], tot[4 * n + 3], a4, a5, a6, a7, b2, b3);
          }
        }
      }
    }
  } else {
    // boxes (row block, K half) of 32 row pairs x 128 K bytes, 128-byte swizzle
    const int pc_shift = (rowA & 1) * 4;  // the rows' nibble (rowA, rowB: same parity)
    const int prA = (rowA & 63) >> 1, prB = (rowB & 63) >> 1;
#pragma unroll
    for (int hh = 0; hh < (FULLK ? 2 : 1); ++hh) {
      const int h = FULLK ? hh : kh;
      const uint8_t* pA = sA + ((rowA >> 6) * 2 + h) * 4096 + prA * 128;
      const uint8_t* pB = sA + ((rowB >> 6) * 2 + h) * 4096 + prB * 128;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int jj = 4 * m + t;  // 16-K chunk of the K half
        const uint4 ca = *reinterpret_cast<const uint4*>(pA + ((jj ^ (prA & 7)) << 4));
        const uint4 cb = *reinterpret_cast<const uint4*>(pB + ((jj ^ (prB & 7)) << 4));
        const uint32_t wa[4] = {ca.x, ca.y, ca.z, ca.w}, wb[4] = {cb.x, cb.y, cb.z, cb.w};
        // code pairs of word i = K 4i .. 4i + 3: (k0, k2), (k1, k3)
        uint32_t a0[4], a1[4], a2[4], a3[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t a = wa[i] >> pc_shift, b = wb[i] >> pc_shift;
          a0[i] = code_pair<DT>(a);
          a1[i] = code_pair<DT>(b);
          a2[i] = code_pair<DT>(a >> 8);
          a3[i] = code_pair<DT>(b >> 8);
        }
#pragma unroll
        for (int n = 0; n < NB; ++n) {
          // activations K 128 h + 16 jj .. + 15 of route 8n + g, paired likewise
          const uint8_t* xp = sX + n * 8 * kGvRouteBytes + (8 * h + jj) * 32;
          const uint4 x0 = *reinterpret_cast<const uint4*>(xp);
          const uint4 x1 = *reinterpret_cast<const uint4*>(xp + 16);
          const uint32_t xb[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
            mma_16816<DT>(tot[4 * n + 0], tot[4 * n + 1], tot[4 * n + 2], tot[4 * n + 3], a0[i], a1[i], a2[i],
                          a3[i], __byte_perm(xb[2 * i], xb[2 * i + 1], 0x5410),
                          __byte_perm(xb[2 * i], xb[2 * i + 1], 0x7632));
        }
      }
    }
  }
}

// Epilogue of one unit on one compute warp; only `fin` warps hold final sums
// and store, every warp takes part in the split-K barriers.
template <int WHICH, int SCALE, int DT, int NB>
__device__ __forceinline__ bool gemv_epilogue(const GemmParams& p, uint64_t* epibar, volatile int* abort_flag,
                                              volatile int* fixup_flag, const GvUnit& w, int e, int m0, int rows,
                                              int rowA, int rowB, int rb, int lane, bool fin, uint32_t& eph,
                                              const float (&tot)[4 * NB]) {
  using T = F16<DT>;
  const int t = lane & 3;
  const bool gated = (WHICH == GEMM_UP && p.act == ACT_SWIGLU);
  const int N1 = p.n_rows;
  int r0, r1;
  tile_row_bases<WHICH>(p, w.nt, r0, r1);
  const int growA = rowA < 64 ? r0 + rowA : r1 + (rowA - 64);  // weight rows in the expert
  const int growB = rowB < 64 ? r0 + rowB : r1 + (rowB - 64);
  const bool okA = gated ? (64 * w.nt + (rowA & 63)) < p.inter : growA < N1;
  const bool okB = gated ? okA : growB < N1;
  float scA = 1.0f, scB = 1.0f;
  if (SCALE == SCALE_CHANNEL) {
    if (okA) scA = bf16_bits_to_float(p.scales[static_cast<int64_t>(e) * N1 + growA]);
    if (okB) scB = bf16_bits_to_float(p.scales[static_cast<int64_t>(e) * N1 + growB]);
  }
  // Bounded barrier over the 16 compute warps.
  auto grp_sync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(epibar);
    const bool ok = warp_wait(epibar, eph & 1, abort_flag, p.err, p.wait_ns);
    ++eph;
    return ok;
  };

  if (WHICH == GEMM_DOWN) {
    if (!fin) return true;
    const int64_t oc = p.out_cols;
    const int64_t y0 = (static_cast<int64_t>(w.split) * p.slots_cap + m0) * oc;
    if (p.out16) {
      // expert outputs in the activation dtype (one rounding)
      uint16_t* y = reinterpret_cast<uint16_t*>(p.out) + y0;
#pragma unroll
      for (int n = 0; n < NB; ++n) {
        const int rt0 = 8 * n + 2 * t, rt1 = rt0 + 1;
        if (rt0 < rows && okA) y[rt0 * oc + growA] = F16<DT>::from_float(tot[4 * n + 0] * scA);
        if (rt1 < rows && okA) y[rt1 * oc + growA] = F16<DT>::from_float(tot[4 * n + 1] * scA);
        if (rt0 < rows && okB) y[rt0 * oc + growB] = F16<DT>::from_float(tot[4 * n + 2] * scB);
        if (rt1 < rows && okB) y[rt1 * oc + growB] = F16<DT>::from_float(tot[4 * n + 3] * scB);
      }
      return true;
    }
    float* y = reinterpret_cast<float*>(p.out) + y0;
#pragma unroll
    for (int n = 0; n < NB; ++n) {
      const int rt0 = 8 * n + 2 * t, rt1 = rt0 + 1;
      if (rt0 < rows && okA) y[rt0 * oc + growA] = tot[4 * n + 0] * scA;
      if (rt1 < rows && okA) y[rt1 * oc + growA] = tot[4 * n + 1] * scA;
      if (rt0 < rows && okB) y[rt0 * oc + growB] = tot[4 * n + 2] * scB;
      if (rt1 < rows && okB) y[rt1 * oc + growB] = tot[4 * n + 3] * scB;
    }
    return true;
  }

  uint16_t* inter = reinterpret_cast<uint16_t*>(p.out) + static_cast<int64_t>(m0) * p.inter;
  if (p.splits > 1) {
    float* part = p.part + (static_cast<int64_t>(w.split) * p.slots_cap + m0) * N1;
#pragma unroll
    for (int n = 0; n < NB; ++n) {
      const int rt0 = 8 * n + 2 * t, rt1 = rt0 + 1;
      if (!fin) break;
      if (rt0 < rows && okA) part[static_cast<int64_t>(rt0) * N1 + growA] = tot[4 * n + 0] * scA;
      if (rt1 < rows && okA) part[static_cast<int64_t>(rt1) * N1 + growA] = tot[4 * n + 1] * scA;
      if (rt0 < rows && okB) part[static_cast<int64_t>(rt0) * N1 + growB] = tot[4 * n + 2] * scB;
      if (rt1 < rows && okB) part[static_cast<int64_t>(rt1) * N1 + growB] = tot[4 * n + 3] * scB;
    }
    // The last split to finish sums the partials in split order
    // (deterministic) and applies the activation.
    __threadfence();
    if (!grp_sync()) return false;
    if (fin && rb == 0 && lane == 0) {
      const int prev = atomicAdd(&p.counters[w.tile * p.n_tiles + w.nt], 1);
      *fixup_flag = (prev == p.splits - 1) ? 1 : 0;
    }
    if (!grp_sync()) return false;
    const bool last = *fixup_flag != 0;
    if (last && fin) {
      __threadfence();
      const int64_t sstride = p.slots_cap * static_cast<int64_t>(N1);
      // lanes t take routes t, t + 4, ... of their rows
      for (int r = t; r < rows; r += 4) {
        const float* src = p.part + static_cast<int64_t>(m0 + r) * N1;
        if (gated) {
          const int i = 64 * w.nt + (rowA & 63);
          if (okA) {
            float gs = 0.0f, us = 0.0f;
            for (int s = 0; s < p.splits; ++s) {
              gs += __ldcg(src + s * sstride + i);
              us += __ldcg(src + s * sstride + p.inter + i);
            }
            inter[static_cast<int64_t>(r) * p.inter + i] = T::from_float(silu_f(gs) * us);
          }
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int gr = h ? growB : growA;
            if (h ? okB : okA) {
              float hs = 0.0f;
              for (int s = 0; s < p.splits; ++s) hs += __ldcg(src + s * sstride + gr);
              const float a = hs > 0.0f ? hs : 0.0f;
              inter[static_cast<int64_t>(r) * p.inter + gr] = T::from_float(a * a);
            }
          }
        }
      }
      if (rb == 0 && lane == 0) p.counters[w.tile * p.n_tiles + w.nt] = 0;
    }
    // the flag is rewritten only after this group's next two barriers
    return true;
  }

  if (!fin) return true;
#pragma unroll
  for (int n = 0; n < NB; ++n) {
    const int rt0 = 8 * n + 2 * t, rt1 = rt0 + 1;
    const float vA0 = tot[4 * n + 0] * scA, vA1 = tot[4 * n + 1] * scA;
    const float vB0 = tot[4 * n + 2] * scB, vB1 = tot[4 * n + 3] * scB;
    if (gated) {
      // rowA = gate row, rowB = its up row (same intermediate index)
      const int i = 64 * w.nt + (rowA & 63);
      if (okA) {
        if (rt0 < rows) inter[static_cast<int64_t>(rt0) * p.inter + i] = T::from_float(silu_f(vA0) * vB0);
        if (rt1 < rows) inter[static_cast<int64_t>(rt1) * p.inter + i] = T::from_float(silu_f(vA1) * vB1);
      }
    } else {
      auto relu2 = [](float h) {
        const float a = h > 0.0f ? h : 0.0f;
        return a * a;
      };
      if (rt0 < rows && okA) inter[static_cast<int64_t>(rt0) * p.inter + growA] = T::from_float(relu2(vA0));
      if (rt1 < rows && okA) inter[static_cast<int64_t>(rt1) * p.inter + growA] = T::from_float(relu2(vA1));
      if (rt0 < rows && okB) inter[static_cast<int64_t>(rt0) * p.inter + growB] = T::from_float(relu2(vB0));
      if (rt1 < rows && okB) inter[static_cast<int64_t>(rt1) * p.inter + growB] = T::from_float(relu2(vB1));
    }
  }
  return true;
}

// One unit on one compute warp of group `grp`.  Units of several stages
// (!alt): the warp computes K half `grp` of every stage and the halves meet in
// the exchange buffer.  Single-stage units (alt): group `grp` takes the units
// of ordinal parity `grp` over the full K, on a ring of its own.
//
// Every consumer of a ring waits on every phase of its slots: a ring is shared
// by all 16 compute warps (!alt), or belongs to one group (alt), whose 8 warps
// are then its only consumers.  Parity waits therefore never see a slot more
// than one phase away, and the producer refills a slot only after all of its
// consumers left it.
template <int WHICH, int SCALE, int DT, int LAYOUT, int NB>
__device__ __forceinline__ bool gemv_unit(const GemmParams& p, uint8_t* smem, uint64_t* full, uint64_t* empty, uint64_t* epibar, volatile int* abort_flag,
                                          volatile int* fixup_flag, float* red, const GvUnit& w, const int4& ti,
                                          bool alt, int grp, int rowA, int rowB, int rb, int lane,
                                          uint32_t ld_row_off, int ld_row7, int ld_chunk, int ring0, int ring_len,
                                          int& st, uint32_t& ph, uint32_t& eph) {
  float tot[4 * NB];
#pragma unroll
  for (int j = 0; j < 4 * NB; ++j) tot[j] = 0.0f;
  for (int kb = w.kb0; kb < w.kb1; ++kb) {
    const int slot = ring0 + st;
    if (!warp_wait(&full[slot], ph, abort_flag, p.err, p.wait_ns)) return false;
    const uint8_t* sA = smem + slot * p.stage_bytes;
    if (alt) gemv_stage<SCALE, DT, LAYOUT, NB, true>(sA, rowA, rowB, grp, lane, ld_row_off, ld_row7, ld_chunk, tot);
    else gemv_stage<SCALE, DT, LAYOUT, NB, false>(sA, rowA, rowB, grp, lane, ld_row_off, ld_row7, ld_chunk, tot);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    ring_next(st, ph, ring_len);
  }
  bool fin = true;
  if (!alt) {
    // K halves meet: group 1 leaves its sums in one of two buffers (alternating
    // per unit: a buffer is rewritten only after every warp passed the next
    // barrier, i.e. after group 0 read it); group 0 adds them and finishes.
    // (buffers of the plan's largest NB, bn / 8: units of different NB never
    // overlap in them)
    float4* rbuf = reinterpret_cast<float4*>(red) + ((eph & 1) * 8 + rb) * (p.bn >> 3) * 32 + lane;
    if (grp == 1) {
#pragma unroll
      for (int n = 0; n < NB; ++n)
        rbuf[n * 32] = make_float4(tot[4 * n + 0], tot[4 * n + 1], tot[4 * n + 2], tot[4 * n + 3]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(epibar);
    if (!warp_wait(epibar, eph & 1, abort_flag, p.err, p.wait_ns)) return false;
    ++eph;
    fin = grp == 0;
    if (fin) {
#pragma unroll
      for (int n = 0; n < NB; ++n) {
        const float4 o = rbuf[n * 32];
        tot[4 * n + 0] += o.x;
        tot[4 * n + 1] += o.y;
        tot[4 * n + 2] += o.z;
        tot[4 * n + 3] += o.w;
      }
    }
  }
  return gemv_epilogue<WHICH, SCALE, DT, NB>(p, epibar, abort_flag, fixup_flag, w, ti.x, ti.y,
                                             min(ti.z, kGemvMaxR), rowA, rowB, rb, lane, fin, eph, tot);
}

template <int WHICH, int SCALE, int DT, int LAYOUT>
__global__ void __launch_bounds__(kGemvThreads, 1)
    w4a16_gemv_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmS) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int stages = p.stages;
  uint8_t* ctrl = smem + stages * p.stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + kGemvMaxStages;
  uint64_t* epibar = empty + kGemvMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(epibar + 1);
  volatile int* fixup_flag = abort_flag + 1;
  volatile int* prod_issued = fixup_flag + 1;  // [2]: stages the producer issued per ring
  volatile int* prod_stopped = prod_issued + 2;
  int4* tile_tab = reinterpret_cast<int4*>(ctrl + kGvCtrlTabOff);
  float* red = reinterpret_cast<float*>(ctrl + kGvCtrlRedOff);
  // single-stage units without split: the compute groups take alternate units,
  // each on a ring of its own (slots [0, ring_len) and [ring_len, 2 ring_len))
  const bool alt = p.splits == 1 && p.kb_total == 1;
  const int ring_len = alt ? stages / 2 : stages;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], kGvFullArrivals);      // producer (TMA bytes) + activation copies
      mbar_init(&empty[s], alt ? kGemvComputeWarps / 2 : kGemvComputeWarps);  // the ring's consumers
    }
    mbar_init(epibar, kGemvComputeWarps);
    *abort_flag = 0;
    *fixup_flag = 0;
    *prod_stopped = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    if (p.scale_tma) tma_prefetch_desc(&tmS);
  }
  __syncthreads();

  // Everything below reads what the previous kernels wrote.
  pdl_wait();
  pdl_launch_dependents();

  // Tile records of this CTA's units blockIdx.x + i * gridDim.x, i < kGemvTileTab,
  // one per thread, loaded together with the tile count (indices clamped to
  // the list's capacity; records past the count are never used).
  if (threadIdx.x < kGemvTileTab) {
    const int64_t u = blockIdx.x + static_cast<int64_t>(threadIdx.x) * gridDim.x;
    const int64_t t = min(u / (p.splits * p.n_tiles), static_cast<int64_t>(p.tiles_cap - 1));
    tile_tab[threadIdx.x] = p.tiles[t];
  }
  const int n_units = (*p.num_tiles) * p.n_tiles * p.splits;
  const int N1 = p.n_rows;
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_s = l2_policy_evict_last();  // each scale sector serves two stages
    const int groups_row = p.K / kGroup;
    const int sbytes_row = groups_row * 2;
    const bool stma = SCALE == SCALE_GROUP && p.scale_tma;
    int st_r0 = 0, st_r1 = 0;
    uint32_t ph_r0 = 0, ph_r1 = 0, issued_r0 = 0, issued_r1 = 0;
    bool ok = true;
    UnitIter it;
    it.init(p);
    for (int i = 0; it.u < n_units && ok; it.next(p), ++i) {
      const GvUnit w = it.unit(p);
      const int4 ti = tile_of(p, tile_tab, i, it.u);
      if (w.kb1 <= w.kb0) continue;
      const int e = ti.x;
      int r0, r1;
      tile_row_bases<WHICH>(p, w.nt, r0, r1);
      const int ring = alt ? (i & 1) : 0;
      int st = ring ? st_r1 : st_r0;
      uint32_t ph = ring ? ph_r1 : ph_r0;
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
        const int slot = ring * ring_len + st;
        if (!warp_wait(&empty[slot], ph ^ 1u, abort_flag, p.err, p.wait_ns)) {
          ok = false;
          break;
        }
        uint8_t* sA = smem + slot * p.stage_bytes;
        uint8_t* sS = sA + kGvOffS;
        if (SCALE == SCALE_GROUP && !stma) {
          // the stage's 8 group scales (16 bytes) of each tile row (lane + 32 j);
          // rows beyond the expert's rows read as zero
          const int g0 = kb * (kGemvBlockK / kGroup);
          const int ng = min(kGemvBlockK / kGroup, groups_row - g0);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int tr = lane + 32 * j;
            const int grow = tr < 64 ? r0 + tr : r1 + (tr - 64);
            uint8_t* dst = sS + tr * kGvScaleRowBytes;
            const uint8_t* src = reinterpret_cast<const uint8_t*>(p.scales) +
                                 (static_cast<int64_t>(e) * N1 + grow) * sbytes_row + g0 * 2;
            static_assert(kGvScaleRowBytes == 16, "one 16-byte scale piece per row and stage");
            copy_scale_piece(dst, src, grow < N1 ? max(ng, 0) * 2 : 0);
          }
          cp_async_mbar_arrive(&full[slot]);
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[slot], kGvWeightBytes + (stma ? kTileRows * kGvScaleRowBytes : 0));
          if (SCALE == SCALE_GROUP || LAYOUT == LAYOUT_IL) {
            // two 64-row boxes of 128 packed bytes (256 K values)
            tma_load_3d(sA, &tmA, &full[slot], kb * (kGemvBlockK / 2), r0, e, pol_w);
            tma_load_3d(sA + 8192, &tmA, &full[slot], kb * (kGemvBlockK / 2), r1, e, pol_w);
            if (stma) {
              // two 64-row boxes of the stage's 8 BF16 scales
              tma_load_3d(sS, &tmS, &full[slot], kb * (kGemvBlockK / kGroup), r0, e, pol_s);
              tma_load_3d(sS + 64 * kGvScaleRowBytes, &tmS, &full[slot], kb * (kGemvBlockK / kGroup), r1, e, pol_s);
            }
          } else {
            // (row block, K half) boxes of 32 row pairs x 128 K bytes
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
              for (int h = 0; h < 2; ++h)
                tma_load_3d(sA + (b * 2 + h) * 4096, &tmA, &full[slot], kb * kGemvBlockK + h * 128,
                            (b ? r1 : r0) / 2, e, pol_w);
          }
        }
        __syncwarp();
        if (ring) ++issued_r1;
        else ++issued_r0;
        ring_next(st, ph, ring_len);
      }
      if (ring) {
        st_r1 = st;
        ph_r1 = ph;
      } else {
        st_r0 = st;
        ph_r0 = ph;
      }
    }
    // Wind-down: publish the stage counts for warp 1 (which owes the stages
    // it did not reach after an abort their arrivals), then wait (bounded)
    // until the copies of the last stages of each ring have landed -- after
    // a normal run the compute warps consumed them all and the waits return
    // at once; after an abort copies may still be in flight.
    if (lane == 0) {
      prod_issued[0] = static_cast<int>(issued_r0);
      prod_issued[1] = static_cast<int>(issued_r1);
      __threadfence_block();
      *prod_stopped = 1;
      volatile int no_abort = 0;
      auto drain = [&](int r, uint32_t n) {
        const uint32_t from = n > static_cast<uint32_t>(ring_len) ? n - ring_len : 0;
        for (uint32_t j = from; j < n; ++j)
          mbar_wait(&full[r * ring_len + j % ring_len], (j / ring_len) & 1, &no_abort, p.err);
      };
      drain(0, issued_r0);
      if (alt) drain(1, issued_r1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ activation rows
    // One route row per pass, 8 K values (16 B) per lane, straight from x (by
    // token) or the intermediate (by slot) with cp.async; out-of-range K is
    // zero-filled by the copy.  Each lane's cp.async.mbarrier.arrive counts as one
    // of the stage's arrivals once its copies have landed; the warp never
    // blocks on them.
    const uint16_t* xsrc = reinterpret_cast<const uint16_t*>(p.x);
    int st_r0 = 0, st_r1 = 0;
    uint32_t ph_r0 = 0, ph_r1 = 0, done_r0 = 0, done_r1 = 0;
    bool ok = true;
    // source row of route `lane` of a tile (lanes below its route count)
    auto src_of = [&](const int4& t) -> int {
      int src = 0;
      if (lane < min(t.z, kGemvMaxR)) {
        if (WHICH == GEMM_UP) {
          const int route = p.perm[t.y + lane];
          src = route >= 0 ? route / p.top_k : 0;
        } else {
          src = t.y + lane;
        }
      }
      return src;
    };
    int src_next = static_cast<int>(blockIdx.x) < n_units ? src_of(tile_tab[0]) : 0;
    UnitIter it;
    it.init(p);
    for (int i = 0; it.u < n_units && ok; it.next(p), ++i) {
      const int u = it.u;
      const GvUnit w = it.unit(p);
      const int4 ti = tile_of(p, tile_tab, i, u);
      const int src = src_next;
      const int rows = min(ti.z, kGemvMaxR);
      const int ring = alt ? (i & 1) : 0;
      int st = ring ? st_r1 : st_r0;
      uint32_t ph = ring ? ph_r1 : ph_r0;
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
        const int slot = ring * ring_len + st;
        if (!warp_wait(&empty[slot], ph ^ 1u, abort_flag, p.err, p.wait_ns)) {
          ok = false;
          break;
        }
        uint8_t* xs = smem + slot * p.stage_bytes + kGvOffX;
        const int col = kb * kGemvBlockK + lane * 8;
        const bool valid = col < p.K;
        for (int r = 0; r < rows; ++r) {
          const int srow = __shfl_sync(0xFFFFFFFFu, src, r);
          cp_async_cg16(xs + r * kGvRouteBytes + lane * 16,
                        xsrc + static_cast<int64_t>(srow) * p.K + (valid ? col : 0), valid ? 16u : 0u);
        }
        cp_async_mbar_arrive_noinc(&full[slot]);
        if (ring) ++done_r1;
        else ++done_r0;
        ring_next(st, ph, ring_len);
      }
      if (ring) {
        st_r1 = st;
        ph_r1 = ph;
      } else {
        st_r0 = st;
        ph_r0 = ph;
      }
      // the next unit's source rows, loaded while this unit streams
      const int u_next = u + G;
      if (u_next < n_units) src_next = src_of(tile_of(p, tile_tab, i + 1, u_next));
    }
    // After an abort: the arrivals owed to stages the producer issued beyond
    // this warp's last one (the producer is at most a ring ahead: a stage is
    // released only after its activation copies).
    if (!ok && lane == 0) {
      const uint64_t t0 = global_timer_ns();
      while (!*prod_stopped && global_timer_ns() - t0 < kWaitTimeoutNs) {
      }
      if (*prod_stopped) {
        __threadfence_block();
        auto owe = [&](int r, uint32_t from, uint32_t to) {
          for (uint32_t j = from; j < to; ++j) mbar_arrive_cnt(&full[r * ring_len + j % ring_len], 32);
        };
        owe(0, done_r0, static_cast<uint32_t>(prod_issued[0]));
        if (alt) owe(1, done_r1, static_cast<uint32_t>(prod_issued[1]));
      }
    }
    // Every copy lands before the CTA exits.
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    // ------------------------------------------------------------------ compute + epilogue
    // warp 2 + c: group c / 8 (K half, or units of that ordinal parity when
    // alt), row block rb = c % 8
    const int cw = warp - 2, grp = cw >> 3, rb = cw & 7, g = lane >> 2;
    const bool gated = (WHICH == GEMM_UP && p.act == ACT_SWIGLU);
    // SwiGLU: MMA row g = gate row, g + 8 = its up row; otherwise 16 consecutive rows
    const int rowA = gated ? 8 * rb + g : 16 * rb + g;
    const int rowB = gated ? 64 + 8 * rb + g : 16 * rb + 8 + g;
    // ldmatrix row of this lane: matrix l / 8 = (rowA or rowB of row l % 8, group
    // offset 0 or 1); byte offset of the row in the stage, its swizzle phase
    const int ld_i = lane & 7, ld_j = lane >> 3;
    const int ld_row = (ld_j & 1) ? rowB - g + ld_i : rowA - g + ld_i;
    const uint32_t ld_row_off = (ld_row >> 6) * 8192 + (ld_row & 63) * 128;
    const int ld_row7 = ld_row & 7, ld_chunk = ld_j >> 1;
    int st = 0;
    uint32_t ph = 0, eph = 0;
    UnitIter it;
    it.init(p);
    const int ring0 = alt ? grp * ring_len : 0;
    for (int i = 0; it.u < n_units; it.next(p), ++i) {
      if (alt && (i & 1) != grp) continue;  // the other group's unit, on the other ring
      const GvUnit w = it.unit(p);
      const int4 ti = tile_of(p, tile_tab, i, it.u);
      const int nb = (min(ti.z, kGemvMaxR) + 7) >> 3;
      bool ok;
#define W4A16_GEMV_UNIT(NBV)                                                                                    \
  gemv_unit<WHICH, SCALE, DT, LAYOUT, NBV>(p, smem, full, empty, epibar, abort_flag, fixup_flag, red, w, ti, alt, \
                                   grp, rowA, rowB, rb, lane, ld_row_off, ld_row7, ld_chunk, ring0, ring_len, st, \
                                   ph, eph)
      if (nb <= 1) ok = W4A16_GEMV_UNIT(1);
      else if (nb == 2) ok = W4A16_GEMV_UNIT(2);
      else ok = W4A16_GEMV_UNIT(4);
#undef W4A16_GEMV_UNIT
      if (!ok) break;
    }
  }
  __syncthreads();
}

template <int WHICH, int SCALE, int DT, int LAYOUT>
cudaError_t launch_gemv_one(const GemmParams& p, const CUtensorMap& tmA, const CUtensorMap& tmS, int grid,
                            int smem_bytes, cudaStream_t s, bool pdl) {
  auto kern = w4a16_gemv_kernel<WHICH, SCALE, DT, LAYOUT>;
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
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, tmA, tmS);
}

template <int DT, int LAYOUT>
cudaError_t launch_gemv_dt(int which, int scale_kind, const GemmParams& p, const CUtensorMap& tmA,
                           const CUtensorMap& tmS, int grid, int smem_bytes, cudaStream_t s, bool pdl) {
  if (which == GEMM_UP) {
    return scale_kind == SCALE_GROUP
               ? launch_gemv_one<GEMM_UP, SCALE_GROUP, DT, LAYOUT>(p, tmA, tmS, grid, smem_bytes, s, pdl)
               : launch_gemv_one<GEMM_UP, SCALE_CHANNEL, DT, LAYOUT>(p, tmA, tmS, grid, smem_bytes, s, pdl);
  }
  return scale_kind == SCALE_GROUP
             ? launch_gemv_one<GEMM_DOWN, SCALE_GROUP, DT, LAYOUT>(p, tmA, tmS, grid, smem_bytes, s, pdl)
             : launch_gemv_one<GEMM_DOWN, SCALE_CHANNEL, DT, LAYOUT>(p, tmA, tmS, grid, smem_bytes, s, pdl);
}

}  // namespace w4a16
