// Expert-grouped W4A16 GEMV for sm_103a (both MoE GEMMs, few routes per
// expert), on warp-level MMAs fed by register-side dequantisation.
//
// Same operation, work units and outputs as the tcgen05 kernel in gemm.cuh
// (route tile x 128-row weight tile x K split; the "gate/up GEMM" and "down
// GEMM" of "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy), sections
// Modification and Benchmark), for batches where an expert sees only a handful
// of routes.  There each weight is used by 1-4 routes: the contraction is a
// matrix-vector product whose cost is streaming the packed INT4 weights, and a
// 128-row tcgen05 tile with TMEM staging has a fixed cost per MMA that such
// thin tiles cannot amortise.  Here the route tile (<= kGemvMaxR = 8 routes)
// is the N = 8 side of mma.sync m16n8k16 and the dequantised weights go to the
// MMA straight from registers.
//
// Arithmetic (per weight row, per 32-element group), in the activation type
// (BF16 or FP16) with FP32 accumulation:
//   * a nibble goes to each 16-bit half of a register with one lop3
//     ((w & 0x000F000F) ^ magic = B + q exactly, B = 136 for BF16 and 1032
//     for FP16, nibble = q & 15) and one HSUB2 of B leaves the exact code q;
//     shifting the word by 4, 8 and 12 bits gives the other three nibble pairs;
//   * the MMA multiplies the exact codes by the activations as given and sums
//     in FP32, one group (two MMAs) at a time; the group result is multiplied
//     by the group scale and accumulated in FP32.
//   Per-channel scales multiply the FP32 total in the epilogue.
//
// A pipeline stage is 128 weight rows x kGemvBlockK (256) K values: 128 bytes
// of every packed row per visit, read by TMA in 128-byte-swizzled boxes.
//
// Warp roles (576 threads):
//   warp 0      TMA producer of the packed weight tile and the group scales
//               (TMA when their rows are 16-byte multiples, else cp.async)
//   warp 1      activation rows: cp.async of the tile's rows (gate/up: token
//               rows of x by slot; down: intermediate rows), completion
//               signalled on the stage's mbarrier without blocking the warp
//   warps 2-17  compute: warp 2 + c takes row block c % 8 (16 rows) and K half
//               c / 8 of every stage; the halves meet once per unit through
//               shared memory.  For SwiGLU a row block holds 8 gate rows and
//               their 8 up rows, so the activation is applied in registers.
#pragma once
#include "gemm.cuh"

namespace w4a16 {

// Stage layout (bytes from the 1024-aligned stage base).
constexpr int kGvWeightBytes = kTileRows * kGemvBlockK / 2;          // packed weights
constexpr int kGvScaleRowBytes = kGemvBlockK / kGroup * 2;            // 8 BF16 scales per row
constexpr int kGvOffS = kGvWeightBytes;
constexpr int kGvOffX = kGvOffS + kTileRows * kGvScaleRowBytes;       // activation rows
constexpr int kGvRouteBytes = kGemvBlockK * 2 + 64;                   // + pad: 64 mod 128
static_assert(kGvOffX + kGemvMaxR * kGvRouteBytes <= kGemvStageBytes, "GEMV stage overflow");
static_assert(kGemvStageBytes % 1024 == 0, "GEMV stages must keep 1024-byte alignment");
constexpr int kGemvComputeWarps = 16;
static_assert(kGemvThreads == 32 * (2 + kGemvComputeWarps), "warp roles");
// Control block: mbarriers and flags; the K-half exchange (two buffers of 8
// warps x 32 lanes x 4 floats) from kGvCtrlRedOff; the tile records of the
// CTA's first kGemvTileTab units from kGvCtrlTabOff.
constexpr int kGvCtrlRedOff = 512;
constexpr int kGvCtrlTabOff = kGvCtrlRedOff + 2 * 8 * 32 * 16;
constexpr int kGemvTileTab = 256;
static_assert(3 * kGemvStages * 8 + 8 + 8 <= kGvCtrlRedOff, "control block");
static_assert(kGvCtrlTabOff + kGemvTileTab * 16 <= kGemvCtrlBytes, "tile table");
static_assert(kGemvTileTab <= kGemvThreads, "one record per thread");

__device__ __forceinline__ void ring_next(int& st, uint32_t& ph) {
  if (++st == kGemvStages) {
    st = 0;
    ph ^= 1u;
  }
}

// Tile record of this CTA's i-th unit u: from the shared table (filled at
// kernel start) or, past its end, from global memory.
__device__ __forceinline__ int4 tile_of(const GemmParams& p, const int4* tab, int i, int u) {
  return i < kGemvTileTab ? tab[i] : load_tile(p, u);
}

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
  __device__ __forceinline__ Unit unit(const GemmParams& p) const {
    Unit w;
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
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  if (DT == DT_BF16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
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

// One unit (route tile x weight tile x K split) on one compute warp: 16 weight
// rows (MMA rows g: rowA, g + 8: rowB) x one K half of every stage x the
// tile's <= 8 routes (MMA columns; columns past the route count read stale
// data and are never stored).  ALT (single-stage units, no split): the warp
// takes both K halves, the two warp groups take alternate units, and no
// cross-warp reduction is needed.
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
//     lane t takes 16-byte chunks t and t + 4 of the K half; word i of a chunk
//     (4 K) gives (k0, k2) and (k1, k3) for one MMA pair.
template <int WHICH, int SCALE, int DT, bool ALT>
__device__ __forceinline__ bool gemv_unit(const GemmParams& p, uint8_t* smem, uint64_t* full,
                                          uint64_t* bfull, uint64_t* empty, uint64_t* epibar,
                                          volatile int* abort_flag, volatile int* fixup_flag,
                                          float* red, const Unit& w, int e, int m0, int rows,
                                          int rowA, int rowB, int rb, int kh, int lane, int& st,
                                          uint32_t& ph, uint32_t& eph) {
  using T = F16<DT>;
  const int g = lane >> 2, t = lane & 3;
  const bool gated = (WHICH == GEMM_UP && p.act == ACT_SWIGLU);
  const int N1 = p.n_rows;
  // tot[0..1]: rowA x routes 2t, 2t + 1; tot[2..3]: rowB x the same routes
  float tot[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  // per-channel: the rows' nibble (rowA and rowB have the same parity)
  const int pc_shift = (rowA & 1) * 4;
  // ldmatrix row of this lane: matrix l / 8 = (rowA or rowB of row l % 8, chunk
  // offset 0 or 1); byte offset of the row in the stage, its swizzle phase
  const int ld_i = lane & 7, ld_j = lane >> 3;
  const int ld_row = (ld_j & 1) ? rowB - g + ld_i : rowA - g + ld_i;
  const uint32_t ld_row_off = (ld_row >> 6) * 8192 + (ld_row & 63) * 128;
  const int ld_row7 = ld_row & 7, ld_chunk = ld_j >> 1;

  for (int kb = w.kb0; kb < w.kb1; ++kb) {
    if (!mbar_wait(&full[st], ph, abort_flag, p.err) || !mbar_wait(&bfull[st], ph, abort_flag, p.err))
      return false;
    const uint8_t* sA = smem + st * kGemvStageBytes;
    const uint8_t* sXr = sA + kGvOffX + g * kGvRouteBytes;  // this lane's B column (route g)
    // K halves of the stage handled by this warp: its own, or both (ALT)
#pragma unroll
    for (int kk = 0; kk < (ALT ? 2 : 1); ++kk) {
      const int khh = ALT ? kk : kh;
      if (SCALE == SCALE_GROUP) {
        const uint2 sa = *reinterpret_cast<const uint2*>(sA + kGvOffS + rowA * kGvScaleRowBytes + khh * 8);
        const uint2 sb = *reinterpret_cast<const uint2*>(sA + kGvOffS + rowB * kGvScaleRowBytes + khh * 8);
        const uint32_t sbase = smem_u32(sA);
  #pragma unroll
        for (int pq = 0; pq < 2; ++pq) {
          // words t of rowA / rowB in groups 4 khh + 2 pq and + 1 (128-byte swizzle:
          // chunk c of row r at c ^ (r & 7))
          uint32_t w4[4];
          ldmatrix_x4(sbase + ld_row_off + ((((4 * khh + 2 * pq) + ld_chunk) ^ ld_row7) << 4), w4[0], w4[1], w4[2],
                      w4[3]);
  #pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int m = 2 * pq + q;
            const int c = 4 * khh + m;  // group of the stage
            const uint32_t wa = w4[2 * q], wb = w4[2 * q + 1];
            // activations K 32c + 8t .. + 7 of route g: (x0 x1) (x2 x3) (x4 x5) (x6 x7),
            // paired as the codes: (x0 x4) (x1 x5) | (x2 x6) (x3 x7)
            const uint4 xv = *reinterpret_cast<const uint4*>(sXr + (4 * c + t) * 16);
            const uint32_t b0 = __byte_perm(xv.x, xv.z, 0x5410), b1 = __byte_perm(xv.x, xv.z, 0x7632);
            const uint32_t b2 = __byte_perm(xv.y, xv.w, 0x5410), b3 = __byte_perm(xv.y, xv.w, 0x7632);
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            mma_16816<DT>(d, code_pair<DT>(wa), code_pair<DT>(wb), code_pair<DT>(wa >> 4), code_pair<DT>(wb >> 4),
                          b0, b1);
            mma_16816<DT>(d, code_pair<DT>(wa >> 8), code_pair<DT>(wb >> 8), code_pair<DT>(wa >> 12),
                          code_pair<DT>(wb >> 12), b2, b3);
            // BF16 group scales of rowA / rowB -> FP32 exactly
            const uint32_t swa = (m < 2) ? sa.x : sa.y, swb = (m < 2) ? sb.x : sb.y;
            const float fa = __uint_as_float((m & 1) ? (swa & 0xFFFF0000u) : (swa << 16));
            const float fb = __uint_as_float((m & 1) ? (swb & 0xFFFF0000u) : (swb << 16));
            tot[0] = fmaf(fa, d[0], tot[0]);
            tot[1] = fmaf(fa, d[1], tot[1]);
            tot[2] = fmaf(fb, d[2], tot[2]);
            tot[3] = fmaf(fb, d[3], tot[3]);
          }
        }
      } else {
        // boxes (row block, K half) of 32 row pairs x 128 K bytes, 128-byte swizzle
        const int prA = (rowA & 63) >> 1, prB = (rowB & 63) >> 1;
        const uint8_t* pA = sA + ((rowA >> 6) * 2 + khh) * 4096 + prA * 128;
        const uint8_t* pB = sA + ((rowB >> 6) * 2 + khh) * 4096 + prB * 128;
  #pragma unroll
        for (int m = 0; m < 2; ++m) {
          const int jj = 4 * m + t;  // 16-K chunk of the K half
          const uint4 ca = *reinterpret_cast<const uint4*>(pA + ((jj ^ (prA & 7)) << 4));
          const uint4 cb = *reinterpret_cast<const uint4*>(pB + ((jj ^ (prB & 7)) << 4));
          // activations of the chunk (K 128 khh + 16 jj .. + 15 of route g)
          const uint8_t* xp = sXr + (8 * khh + jj) * 32;
          const uint4 x0 = *reinterpret_cast<const uint4*>(xp);
          const uint4 x1 = *reinterpret_cast<const uint4*>(xp + 16);
          const uint32_t wa[4] = {ca.x, ca.y, ca.z, ca.w}, wb[4] = {cb.x, cb.y, cb.z, cb.w};
          const uint32_t xb[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
  #pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t a = wa[i] >> pc_shift, b = wb[i] >> pc_shift;
            // word i = K 4i .. 4i + 3: code pairs (k0, k2), (k1, k3); activations likewise
            mma_16816<DT>(tot, code_pair<DT>(a), code_pair<DT>(b), code_pair<DT>(a >> 8), code_pair<DT>(b >> 8),
                          __byte_perm(xb[2 * i], xb[2 * i + 1], 0x5410),
                          __byte_perm(xb[2 * i], xb[2 * i + 1], 0x7632));
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    ring_next(st, ph);
  }

  // ---------------------------------------------------------------- epilogue
  auto epi_sync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(epibar);
    const bool ok = mbar_wait(epibar, eph & 1, abort_flag, p.err);
    ++eph;
    return ok;
  };
  // K halves meet: the second half's warps leave their sums in one of two
  // buffers (alternating per unit: a buffer is rewritten only after every warp
  // passed the next barrier, i.e. after the first half read it).
  bool fin = true;  // this warp finishes the unit
  if (!ALT) {
    float4* rbuf = reinterpret_cast<float4*>(red) + ((eph & 1) * 8 + rb) * 32 + lane;
    if (kh == 1) *rbuf = make_float4(tot[0], tot[1], tot[2], tot[3]);
    if (!epi_sync()) return false;
    fin = kh == 0;  // the first half finishes the unit
    if (fin) {
      const float4 o = *rbuf;
      tot[0] += o.x;
      tot[1] += o.y;
      tot[2] += o.z;
      tot[3] += o.w;
    }
  }
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
  const float vA0 = tot[0] * scA, vA1 = tot[1] * scA, vB0 = tot[2] * scB, vB1 = tot[3] * scB;
  const int rt0 = 2 * t, rt1 = 2 * t + 1;  // this lane's routes

  if (WHICH == GEMM_DOWN) {
    if (fin) {
      float* y = reinterpret_cast<float*>(p.out) + (static_cast<int64_t>(w.split) * p.slots_cap + m0) * p.out_cols;
      const int64_t oc = p.out_cols;
      if (rt0 < rows && okA) y[rt0 * oc + growA] = vA0;
      if (rt1 < rows && okA) y[rt1 * oc + growA] = vA1;
      if (rt0 < rows && okB) y[rt0 * oc + growB] = vB0;
      if (rt1 < rows && okB) y[rt1 * oc + growB] = vB1;
    }
    return true;
  }

  uint16_t* inter = reinterpret_cast<uint16_t*>(p.out) + static_cast<int64_t>(m0) * p.inter;
  if (p.splits > 1) {
    if (fin) {
      float* part = p.part + (static_cast<int64_t>(w.split) * p.slots_cap + m0) * N1;
      if (rt0 < rows && okA) part[static_cast<int64_t>(rt0) * N1 + growA] = vA0;
      if (rt1 < rows && okA) part[static_cast<int64_t>(rt1) * N1 + growA] = vA1;
      if (rt0 < rows && okB) part[static_cast<int64_t>(rt0) * N1 + growB] = vB0;
      if (rt1 < rows && okB) part[static_cast<int64_t>(rt1) * N1 + growB] = vB1;
    }
    // The last split to finish sums the partials in split order
    // (deterministic) and applies the activation.
    __threadfence();
    if (!epi_sync()) return false;
    if (rb == 0 && kh == 0 && lane == 0) {
      const int prev = atomicAdd(&p.counters[w.tile * p.n_tiles + w.nt], 1);
      *fixup_flag = (prev == p.splits - 1) ? 1 : 0;
    }
    if (!epi_sync()) return false;
    const bool last = *fixup_flag != 0;
    if (last && fin) {
      __threadfence();
      const int64_t sstride = p.slots_cap * static_cast<int64_t>(N1);
      // lanes t take routes t and t + 4 of their rows
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
    }
    if (last && rb == 0 && kh == 0 && lane == 0) p.counters[w.tile * p.n_tiles + w.nt] = 0;
    return true;
  }

  if (fin) {
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

template <int WHICH, int SCALE, int DT>
__global__ void __launch_bounds__(kGemvThreads, 1)
    w4a16_gemv_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmS) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ctrl = smem + kGemvStages * kGemvStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* bfull = full + kGemvStages;
  uint64_t* empty = bfull + kGemvStages;
  uint64_t* epibar = empty + kGemvStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(epibar + 1);
  volatile int* fixup_flag = abort_flag + 1;
  float* red = reinterpret_cast<float*>(ctrl + kGvCtrlRedOff);
  int4* tile_tab = reinterpret_cast<int4*>(ctrl + kGvCtrlTabOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemvStages; ++s) {
      mbar_init(&full[s], 1);                  // producer (TMA bytes + scale copies)
      mbar_init(&bfull[s], 32);                // the 32 lanes' activation copies
      // every compute warp, or one warp group of 8 when the groups take
      // alternate single-stage units
      mbar_init(&empty[s], (p.splits == 1 && p.kb_total == 1) ? kGemvComputeWarps / 2 : kGemvComputeWarps);
    }
    mbar_init(epibar, kGemvComputeWarps);
    *abort_flag = 0;
    *fixup_flag = 0;
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
    int st = 0;
    uint32_t ph = 0, issued = 0;
    bool ok = true;
    UnitIter it;
    it.init(p);
    for (int i = 0; it.u < n_units && ok; it.next(p), ++i) {
      const Unit w = it.unit(p);
      const int4 ti = tile_of(p, tile_tab, i, it.u);
      if (w.kb1 <= w.kb0) continue;
      const int e = ti.x;
      int r0, r1;
      tile_row_bases<WHICH>(p, w.nt, r0, r1);
      // scale rows of this unit for this lane's tile rows (lane + 32 i); null
      // when the row lies beyond the expert's rows
      const uint8_t* srow[4];
      bool srow_al16 = true;
      if (SCALE == SCALE_GROUP && !p.scale_tma) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int tr = lane + 32 * j;
          const int grow = tr < 64 ? r0 + tr : r1 + (tr - 64);
          srow[j] = grow < N1 ? reinterpret_cast<const uint8_t*>(p.scales) +
                                    (static_cast<int64_t>(e) * N1 + grow) * sbytes_row
                              : nullptr;
          srow_al16 = srow_al16 && ((reinterpret_cast<uintptr_t>(srow[j]) & 15) == 0);
        }
      }
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
        if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        uint8_t* sA = smem + st * kGemvStageBytes;
        uint8_t* sS = sA + kGvOffS;
        if (SCALE == SCALE_GROUP && !p.scale_tma) {
          // the stage's 8 group scales (16 bytes) of each tile row
          const int g0 = kb * (kGemvBlockK / kGroup);
          const int ng = min(kGemvBlockK / kGroup, groups_row - g0);
          if (srow_al16 && ng == kGemvBlockK / kGroup) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint8_t* dst = sS + (lane + 32 * j) * kGvScaleRowBytes;
              if (srow[j]) cp_async_cg16(dst, srow[j] + g0 * 2, 16u);
              else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint8_t* dst = sS + (lane + 32 * j) * kGvScaleRowBytes;
              const int nbytes = srow[j] ? max(ng, 0) * 2 : 0;
              for (int o = 0; o < nbytes; o += 4) cp_async<4>(dst + o, srow[j] + g0 * 2 + o);
              for (int o = nbytes; o < kGvScaleRowBytes; o += 4) *reinterpret_cast<uint32_t*>(dst + o) = 0u;
            }
          }
          cp_async_mbar_arrive(&full[st]);
        }
        __syncwarp();
        if (lane == 0) {
          const bool stma = SCALE == SCALE_GROUP && p.scale_tma;
          mbar_arrive_expect_tx(&full[st], kGvWeightBytes + (stma ? kTileRows * kGvScaleRowBytes : 0));
          if (SCALE == SCALE_GROUP) {
            // two 64-row boxes of 128 packed bytes (256 K values)
            tma_load_3d(sA, &tmA, &full[st], kb * (kGemvBlockK / 2), r0, e, pol_w);
            tma_load_3d(sA + 8192, &tmA, &full[st], kb * (kGemvBlockK / 2), r1, e, pol_w);
            if (stma) {
              // two 64-row boxes of the stage's 8 BF16 scales
              tma_load_3d(sS, &tmS, &full[st], kb * (kGemvBlockK / kGroup), r0, e, pol_s);
              tma_load_3d(sS + 64 * kGvScaleRowBytes, &tmS, &full[st], kb * (kGemvBlockK / kGroup), r1, e, pol_s);
            }
          } else {
            // (row block, K half) boxes of 32 row pairs x 128 K bytes
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
              for (int h = 0; h < 2; ++h)
                tma_load_3d(sA + (b * 2 + h) * 4096, &tmA, &full[st], kb * kGemvBlockK + h * 128,
                            (b ? r1 : r0) / 2, e, pol_w);
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
    // ------------------------------------------------------------------ activation rows
    // One route row per pass, 8 K values (16 B) per lane, straight from x (by
    // token) or the intermediate (by slot) with cp.async; out-of-range K is
    // zero-filled by the copy.  Each lane's cp.async.mbarrier.arrive marks the
    // stage's bfull once its copies have landed; the warp never blocks on them.
    const uint16_t* xsrc = reinterpret_cast<const uint16_t*>(p.x);
    int st = 0;
    uint32_t ph = 0;
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
      const Unit w = it.unit(p);
      const int4 ti = tile_of(p, tile_tab, i, u);
      const int src = src_next;
      const int rows = min(ti.z, kGemvMaxR);
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
        if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        uint8_t* xs = smem + st * kGemvStageBytes + kGvOffX;
        const int col = kb * kGemvBlockK + lane * 8;
        const bool valid = col < p.K;
        for (int r = 0; r < rows; ++r) {
          const int srow = __shfl_sync(0xFFFFFFFFu, src, r);
          cp_async_cg16(xs + r * kGvRouteBytes + lane * 16,
                        xsrc + static_cast<int64_t>(srow) * p.K + (valid ? col : 0), valid ? 16u : 0u);
        }
        cp_async_mbar_arrive_noinc(&bfull[st]);
        ring_next(st, ph);
      }
      // the next unit's source rows, loaded while this unit streams
      const int u_next = u + static_cast<int>(gridDim.x);
      if (u_next < n_units) src_next = src_of(tile_of(p, tile_tab, i + 1, u_next));
    }
    // Every copy lands before the CTA exits (bounded by the compute warps'
    // waits on bfull; the final barrier below follows them).
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    // ------------------------------------------------------------------ compute + epilogue
    // warp 2 + c: row block rb = c % 8 (16 MMA rows), K half kh = c / 8
    const int cw = warp - 2, rb = cw & 7, kh = cw >> 3, g = lane >> 2;
    const bool gated = (WHICH == GEMM_UP && p.act == ACT_SWIGLU);
    // SwiGLU: MMA row g = gate row, g + 8 = its up row; otherwise 16 consecutive rows
    const int rowA = gated ? 8 * rb + g : 16 * rb + g;
    const int rowB = gated ? 64 + 8 * rb + g : 16 * rb + 8 + g;
    // single-stage units without split: the groups (kh) take alternate units
    const bool alt = p.splits == 1 && p.kb_total == 1;
    int st = 0;
    uint32_t ph = 0, eph = 0;
    UnitIter it;
    it.init(p);
    for (int i = 0; it.u < n_units; it.next(p), ++i) {
      if (alt && (i & 1) != kh) {  // the other group's unit: skip its one stage
        ring_next(st, ph);
        continue;
      }
      const Unit w = it.unit(p);
      const int4 ti = tile_of(p, tile_tab, i, it.u);
      const int rows = min(ti.z, kGemvMaxR);
      const bool ok =
          alt ? gemv_unit<WHICH, SCALE, DT, true>(p, smem, full, bfull, empty, epibar, abort_flag, fixup_flag, red,
                                                  w, ti.x, ti.y, rows, rowA, rowB, rb, kh, lane, st, ph, eph)
              : gemv_unit<WHICH, SCALE, DT, false>(p, smem, full, bfull, empty, epibar, abort_flag, fixup_flag, red,
                                                   w, ti.x, ti.y, rows, rowA, rowB, rb, kh, lane, st, ph, eph);
      if (!ok) break;
    }
  }
  __syncthreads();
}

template <int WHICH, int SCALE, int DT>
cudaError_t launch_gemv_one(const GemmParams& p, const CUtensorMap& tmA, const CUtensorMap& tmS, int grid,
                            cudaStream_t s, bool pdl) {
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
  return cudaLaunchKernelEx(&cfg, kern, p, tmA, tmS);
}

template <int DT>
cudaError_t launch_gemv_dt(int which, int scale_kind, const GemmParams& p, const CUtensorMap& tmA,
                           const CUtensorMap& tmS, int grid, cudaStream_t s, bool pdl) {
  if (which == GEMM_UP) {
    return scale_kind == SCALE_GROUP ? launch_gemv_one<GEMM_UP, SCALE_GROUP, DT>(p, tmA, tmS, grid, s, pdl)
                                     : launch_gemv_one<GEMM_UP, SCALE_CHANNEL, DT>(p, tmA, tmS, grid, s, pdl);
  }
  return scale_kind == SCALE_GROUP ? launch_gemv_one<GEMM_DOWN, SCALE_GROUP, DT>(p, tmA, tmS, grid, s, pdl)
                                   : launch_gemv_one<GEMM_DOWN, SCALE_CHANNEL, DT>(p, tmA, tmS, grid, s, pdl);
}

}  // namespace w4a16
