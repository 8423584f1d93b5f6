// Both expert GEMMs of a decode-sized batch in one launch on the CUDA-core
// path (sm_103a): gate/up GEMM + activation, then the down GEMM, fed from one
// device-side work queue.
//
// Same operation as the two launches of gemv.cuh (the "gate/up GEMM" and
// "down GEMM" of "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy),
// sections Modification and Benchmark; the same stage arithmetic,
// gemv_stage), for the batches where an expert sees only a few routes and
// every expert's weights are streamed once.  There two separate launches lose
// time twice: the second launch starts only after the last gate/up unit of
// the first has finished (a whole second wave of long gate/up units runs on
// part of the SMs while the others idle), and every launch pays its own ramp
// (tile records, first weight bytes).  Here every CTA takes queue entries in
// order -- all gate/up units first, then the down units -- so SMs that run
// out of gate/up work stream down weights at once; a down unit needs only the
// intermediate rows of its route tile, which its activation warp waits for
// (the weight bytes are fetched meanwhile).
//
// Queue (one atomic head per forward, zeroed by route preparation):
//   entries [0, Q1):   gate/up units (route tile m, weight tile nt, K split s),
//                      m-major, Q1 = tiles x nt1 x S1
//   entries [Q1, Qt):  down entries (route tile m, down_chunk consecutive
//                      weight tiles), m-major
// Every unit is computed whole by one CTA (split-K partials are summed in
// split order by the last split), so the result does not depend on which CTA
// took which entry: forwards are bit-identical.
//
// No CTA waits for an entry that no running CTA holds: a down entry is taken
// only after every gate/up entry has been taken, a CTA issues its entries in
// the order it took them, and gate/up work never waits on other CTAs.  So the
// grid needs no co-residency, and every wait is bounded all the same.
//
// Pipeline: one ring of stages (weights by TMA, scales, activation rows) with
// an even length; the compute warps form two groups of 8 and group g consumes
// the stages of parity g (each warp: 16 weight rows over the stage's 256 K
// values).  A unit of several stages is split between the groups; at its end
// the group holding the unit's last stage (the finisher) adds the other
// group's sums from a double-buffered exchange and runs the epilogue.  Each
// stage carries a header (unit, K block, tile record) written by the producer.
//
// One-group form (enough gate/up units, no fused finalize; the host
// decides): 320 threads -- the producer, one activation
// warp taking every stage, one compute group of 8 warps that runs every stage
// of its units (no exchange) -- and two CTAs per SM, each with its own ring of
// half the shared memory.  A group's epilogue then holds up only its own ring.
//
// Warp roles (608 threads):
//   warp 0      producer (one lane when every scale row comes by TMA): takes
//               queue entries, writes stage headers, TMA of the weight tile
//               (and of the scales unless the activation warps issue them;
//               cp.async by the whole warp for unaligned scale rows)
//   warp 1      activation rows of the even stages (of every stage with the
//               fused finalize): reads the stage's header; gate/up: token rows
//               of x by route; down: the route tile's intermediate rows, after
//               waiting until all of its gate/up row blocks are published;
//               issues the stage's group-scale TMA when both GEMMs load
//               scales by TMA
//   warps 2-17  compute groups 0 and 1 (row block = warp index mod 8)
//   warp 18     activation rows of the odd stages, or with the fused finalize
//               the finalize warp
//
// Epilogue signals: each finishing warp publishes its 16 intermediate rows of
// route tile m with a release increment of ready[m] (8 row blocks x nt1 weight
// tiles per route tile); with split-K, per-(m, nt, row block) counters elect
// the last split's warp, which sums the FP32 partials in split order.
#pragma once
#include <type_traits>

#include "gemv.cuh"

namespace w4a16 {

constexpr int kItemUp = 0;
constexpr int kItemDown = 1;
constexpr int kItemEnd = 2;

// Stage header (written by the producer, read by the activation warp and the
// compute group of the stage).
struct StageHdr {
  int32_t type, m, nt, kb;         // unit kind, route tile, weight tile, K block
  int32_t e, m0, rows, split;      // tile record (expert, first slot, routes), K split
  uint32_t first_seq, last_seq;    // stage sequence numbers of the unit's first and last stage
  int32_t pad[6];
};
static_assert(sizeof(StageHdr) == 64, "header size");

// Control block of the fused kernel: mbarriers full / empty / hdr per slot,
// the exchange barriers, flags, then the stage headers; the exchange buffers
// follow at kGemvCtrlBytes as in gemv.cuh.
constexpr int kFzOffFull = 0;
constexpr int kFzOffEmpty = kFzOffFull + 8 * kGemvMaxStages;
constexpr int kFzOffHdrBar = kFzOffEmpty + 8 * kGemvMaxStages;
constexpr int kFzOffXBar = kFzOffHdrBar + 8 * kGemvMaxStages;  // xfull[2], xempty[2]
constexpr int kFzOffFlags = kFzOffXBar + 32;                    // abort, issued, stopped
constexpr int kFzOffHdr = 512;
static_assert(kFzOffFlags + 16 <= kFzOffHdr, "control block");
// Fused finalize: a queue of finished (slot range, 16-column block) records
// from the compute warps to the finalize warp.
constexpr int kFinQ = 128;
constexpr int kFzOffFinRec = kFzOffHdr + kGemvMaxStages * 64;  // int4 [kFinQ]
constexpr int kFzOffFinFlag = kFzOffFinRec + kFinQ * 16;       // int [kFinQ]
constexpr int kFzOffFinCtl = kFzOffFinFlag + kFinQ * 4;        // tail, head, done
static_assert(kFzOffFinCtl + 16 <= kGemvCtrlBytes, "finalize queue");
// Warps: producer, activation rows, 16 compute, finalize.
constexpr int kFusedThreads = 32 * (2 + kGemvComputeWarps + 1);
constexpr int kFinWarp = 2 + kGemvComputeWarps;
// One-group form (8-route tiles without the fused finalize): producer,
// activation warp and one compute group of 8 warps, two CTAs per SM.
constexpr int kFusedThreads1 = 32 * (2 + kGemvComputeWarps / 2);
__host__ __device__ constexpr int fused_threads(int groups) { return groups == 1 ? kFusedThreads1 : kFusedThreads; }

// The queue's parts at fixed offsets of the control block (one base pointer:
// every compute warp carries it, and registers are scarce there).
struct FinQueue {
  uint8_t* c;  // the control block
  // records (first slot, routes, first output column, 0)
  __device__ __forceinline__ int4* rec() const { return reinterpret_cast<int4*>(c + kFzOffFinRec); }
  // record i is ready when flag[i % kFinQ] == i + 1
  __device__ __forceinline__ volatile int* flag() const { return reinterpret_cast<volatile int*>(c + kFzOffFinFlag); }
  // records allocated (shared-memory atomic)
  __device__ __forceinline__ int* tail() const { return reinterpret_cast<int*>(c + kFzOffFinCtl); }
  // records consumed by the finalize warp
  __device__ __forceinline__ volatile int* head() const { return reinterpret_cast<volatile int*>(c + kFzOffFinCtl + 4); }
  // compute warps finished
  __device__ __forceinline__ int* done() const { return reinterpret_cast<int*>(c + kFzOffFinCtl + 8); }
};

// A compute warp's last down unit, published one unit later (its fence then
// finds those stores long completed).
struct FinPending {
  int m0, rows, c0;
  bool valid;
};

__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Publish the calling warp's earlier global stores (ordered by __syncwarp)
// with a release increment of *ctr.
__device__ __forceinline__ void warp_publish(int32_t* ctr, int lane) {
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    atomicAdd(ctr, 1);
  }
  __syncwarp();
}

// Epilogue of a gate/up unit on one finishing warp (row block rb): the
// activation of the summed rows into the intermediate, or the FP32 partial of
// this split and, on the last split, the sum of all partials in split order.
template <int SCALE, int DT, int NB>
__device__ __forceinline__ void fused_up_epilogue(const FusedParams& fp, const StageHdr& h, int rowA, int rowB,
                                                  int rb, int lane, const float (&tot)[4 * NB]) {
  using T = F16<DT>;
  const GemmParams& p = fp.up;
  const int t = lane & 3;
  const bool gated = p.act == ACT_SWIGLU;
  const int N1 = p.n_rows;
  const int rows = min(h.rows, kGemvMaxR);
  int r0, r1;
  tile_row_bases<GEMM_UP>(p, h.nt, r0, r1);
  const int growA = rowA < 64 ? r0 + rowA : r1 + (rowA - 64);
  const int growB = rowB < 64 ? r0 + rowB : r1 + (rowB - 64);
  const bool okA = gated ? (64 * h.nt + (rowA & 63)) < p.inter : growA < N1;
  const bool okB = gated ? okA : growB < N1;
  float scA = 1.0f, scB = 1.0f;
  if (SCALE == SCALE_CHANNEL) {
    if (okA) scA = bf16_bits_to_float(p.scales[static_cast<int64_t>(h.e) * N1 + growA]);
    if (okB) scB = bf16_bits_to_float(p.scales[static_cast<int64_t>(h.e) * N1 + growB]);
  }
  uint16_t* inter = reinterpret_cast<uint16_t*>(p.out) + static_cast<int64_t>(h.m0) * p.inter;
  auto relu2 = [](float v) {
    const float a = v > 0.0f ? v : 0.0f;
    return a * a;
  };
  if (p.splits == 1) {
#pragma unroll
    for (int n = 0; n < NB; ++n) {
      const int rt0 = 8 * n + 2 * t, rt1 = rt0 + 1;
      const float vA0 = tot[4 * n + 0] * scA, vA1 = tot[4 * n + 1] * scA;
      const float vB0 = tot[4 * n + 2] * scB, vB1 = tot[4 * n + 3] * scB;
      if (gated) {
        const int i = 64 * h.nt + (rowA & 63);
        if (okA) {
          if (rt0 < rows) inter[static_cast<int64_t>(rt0) * p.inter + i] = T::from_float(silu_f(vA0) * vB0);
          if (rt1 < rows) inter[static_cast<int64_t>(rt1) * p.inter + i] = T::from_float(silu_f(vA1) * vB1);
        }
      } else {
        if (rt0 < rows && okA) inter[static_cast<int64_t>(rt0) * p.inter + growA] = T::from_float(relu2(vA0));
        if (rt1 < rows && okA) inter[static_cast<int64_t>(rt1) * p.inter + growA] = T::from_float(relu2(vA1));
        if (rt0 < rows && okB) inter[static_cast<int64_t>(rt0) * p.inter + growB] = T::from_float(relu2(vB0));
        if (rt1 < rows && okB) inter[static_cast<int64_t>(rt1) * p.inter + growB] = T::from_float(relu2(vB1));
      }
    }
    warp_publish(fp.ready + h.m, lane);
    return;
  }
  // split-K: this split's scaled sums, then the arrival of this row block
  float* part = p.part + (static_cast<int64_t>(h.split) * p.slots_cap + h.m0) * N1;
#pragma unroll
  for (int n = 0; n < NB; ++n) {
    const int rt0 = 8 * n + 2 * t, rt1 = rt0 + 1;
    if (rt0 < rows && okA) part[static_cast<int64_t>(rt0) * N1 + growA] = tot[4 * n + 0] * scA;
    if (rt1 < rows && okA) part[static_cast<int64_t>(rt1) * N1 + growA] = tot[4 * n + 1] * scA;
    if (rt0 < rows && okB) part[static_cast<int64_t>(rt0) * N1 + growB] = tot[4 * n + 2] * scB;
    if (rt1 < rows && okB) part[static_cast<int64_t>(rt1) * N1 + growB] = tot[4 * n + 3] * scB;
  }
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    __threadfence();
    const int prev = atomicAdd(fp.fix + (static_cast<int64_t>(h.m) * p.n_tiles + h.nt) * 8 + rb, 1);
    last = prev == p.splits - 1;
    if (last) __threadfence();
  }
  last = __shfl_sync(0xFFFFFFFFu, last, 0);
  if (!last) return;
  __syncwarp();  // lane 0's acquire orders the other lanes' loads
  // the last split of this row block: partials of every split, summed in split
  // order (all loads of a route issued before the sums)
  const int64_t sstride = p.slots_cap * static_cast<int64_t>(N1);
  const float* src0 = p.part + static_cast<int64_t>(h.m0) * N1;
#pragma unroll
  for (int n = 0; n < NB; ++n) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int rt = 8 * n + 2 * t + c;
      if (rt >= rows) continue;
      const float* src = src0 + static_cast<int64_t>(rt) * N1;
      float a[kMaxFusedSplits], b[kMaxFusedSplits];
#pragma unroll
      for (int s = 0; s < kMaxFusedSplits; ++s) {
        a[s] = (s < p.splits && okA) ? __ldcg(src + s * sstride + growA) : 0.0f;
        b[s] = (s < p.splits && okB) ? __ldcg(src + s * sstride + growB) : 0.0f;
      }
      float sa = 0.0f, sb = 0.0f;
#pragma unroll
      for (int s = 0; s < kMaxFusedSplits; ++s) {
        if (s < p.splits) {
          sa += a[s];
          sb += b[s];
        }
      }
      if (gated) {
        if (okA) inter[static_cast<int64_t>(rt) * p.inter + 64 * h.nt + (rowA & 63)] = T::from_float(silu_f(sa) * sb);
      } else {
        if (okA) inter[static_cast<int64_t>(rt) * p.inter + growA] = T::from_float(relu2(sa));
        if (okB) inter[static_cast<int64_t>(rt) * p.inter + growB] = T::from_float(relu2(sb));
      }
    }
  }
  if (lane == 0) fp.fix[(static_cast<int64_t>(h.m) * p.n_tiles + h.nt) * 8 + rb] = 0;
  warp_publish(fp.ready + h.m, lane);
}

// Output columns [c0, c0 + 16) of token t: its routes' expert outputs in
// top-k order, acc = acc + w * y with two roundings (the combine's arithmetic,
// so the result is bit-identical to the separate combine launch).
template <int DT>
__device__ __forceinline__ void finalize_block(const FusedParams& fp, int t, int c0) {
  const int k = fp.k, H = fp.down.out_cols;
  const float* tw = fp.topk_weights + static_cast<int64_t>(t) * k;
  const int32_t* inv = fp.inv + static_cast<int64_t>(t) * k;
  float wsum = 0.0f;
  if (fp.renormalize)
    for (int j = 0; j < k; ++j) wsum = __fadd_rn(wsum, tw[j]);
  float acc[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) acc[c] = 0.0f;
  const uint16_t* y = reinterpret_cast<const uint16_t*>(fp.down.out);
  // routes in chunks of 4: every load of a chunk is issued before its sums
  // (which stay in top-k order)
  for (int j0 = 0; j0 < k; j0 += 4) {
    int slot[4];
    float w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      slot[i] = j0 + i < k ? inv[j0 + i] : -1;
      w[i] = j0 + i < k ? tw[j0 + i] : 0.0f;
    }
    uint4 u[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (slot[i] >= 0) {
        const uint4* yr = reinterpret_cast<const uint4*>(y + static_cast<int64_t>(slot[i]) * H + c0);
        u[i][0] = __ldcg(yr);
        u[i][1] = __ldcg(yr + 1);
      } else {
        u[i][0] = u[i][1] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (slot[i] < 0) continue;
      float wi = w[i];
      if (fp.renormalize) wi = (wsum != 0.0f) ? __fdiv_rn(wi, wsum) : 0.0f;
      const uint32_t v[8] = {u[i][0].x, u[i][0].y, u[i][0].z, u[i][0].w, u[i][1].x, u[i][1].y, u[i][1].z, u[i][1].w};
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        acc[2 * c] = __fadd_rn(acc[2 * c], __fmul_rn(wi, F16<DT>::to_float(static_cast<uint16_t>(v[c] & 0xFFFFu))));
        acc[2 * c + 1] =
            __fadd_rn(acc[2 * c + 1], __fmul_rn(wi, F16<DT>::to_float(static_cast<uint16_t>(v[c] >> 16))));
      }
    }
  }
  uint32_t o[8];
#pragma unroll
  for (int c = 0; c < 8; ++c)
    o[c] = static_cast<uint32_t>(F16<DT>::from_float(acc[2 * c])) |
           (static_cast<uint32_t>(F16<DT>::from_float(acc[2 * c + 1])) << 16);
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(fp.out) + static_cast<int64_t>(t) * H + c0);
  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// Publish a compute warp's pending record: every lane's fence makes its output
// stores visible to the device, then lane 0 queues the record for the finalize
// warp (waiting, bounded, for a free entry).
__device__ __forceinline__ bool fin_publish(const FusedParams& fp, const FinQueue& fq, FinPending& pend, int lane,
                                            volatile int* abort_flag) {
  __threadfence();
  __syncwarp();
  int ok = 1;
  if (lane == 0) {
    const int i = atomicAdd(fq.tail(), 1);
    const uint64_t t0 = global_timer_ns();
    while (i - *fq.head() >= kFinQ) {
      if (*abort_flag) {
        ok = 0;
        break;
      }
      if (global_timer_ns() - t0 > fp.up.wait_ns) {
        *abort_flag = 1;
        atomicExch(fp.up.err, kErrTimeout);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    if (ok) {
      fq.rec()[i % kFinQ] = make_int4(pend.m0, pend.rows, pend.c0, 0);
      __threadfence_block();
      fq.flag()[i % kFinQ] = i + 1;
    }
  }
  pend.valid = false;
  return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// The finalize warp: takes ready records in order, up to 32 routes at a time
// (one lane per route); per route one arrival on its (token, 16-column block)
// counter; the arrival that completes a token's valid routes sums the block.
template <int DT>
__device__ __forceinline__ void fin_warp(const FusedParams& fp, const FinQueue& fq, int lane,
                                         volatile int* abort_flag) {
  const GemmParams& p = fp.down;
  const int nblk = p.n_rows / 16;
  int head = 0;
  const uint64_t t0 = global_timer_ns();
  uint64_t last_progress = t0;
  for (;;) {
    const int idx = head + lane;
    const bool rdy = fq.flag()[idx % kFinQ] == idx + 1;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, rdy);
    const int n = (m == 0xFFFFFFFFu) ? 32 : __ffs(~m) - 1;  // ready records in order
    if (n == 0) {
      if (*fq.done() == kGemvComputeWarps && *reinterpret_cast<volatile int*>(fq.tail()) == head) break;
      if (*abort_flag) break;
      if (global_timer_ns() - last_progress > fp.up.wait_ns) {
        if (lane == 0) {
          *abort_flag = 1;
          atomicExch(fp.up.err, kErrTimeout);
        }
        break;
      }
      __nanosleep(64);
      continue;
    }
    __threadfence_block();
    const int4 rec = lane < n ? fq.rec()[idx % kFinQ] : make_int4(0, 0, 0, 0);
    // records whose routes fit in this pass (every record holds <= 32 routes)
    int incl = rec.y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    const int ex = incl - rec.y;
    const int taken = __popc(__ballot_sync(0xFFFFFFFFu, lane < n && incl <= 32));
    const int total = __shfl_sync(0xFFFFFFFFu, incl, taken - 1);
    // lane -> (record j, route r)
    int j = 0;
    for (int i = 1; i < taken; ++i)
      if (__shfl_sync(0xFFFFFFFFu, ex, i) <= lane) j = i;
    const int m0 = __shfl_sync(0xFFFFFFFFu, rec.x, j);
    const int c0 = __shfl_sync(0xFFFFFFFFu, rec.z, j);
    const int r = lane - __shfl_sync(0xFFFFFFFFu, ex, j);
    int fin_t = -1;
    if (lane < total) {
      const int route = p.perm[m0 + r];
      const int t = route / fp.k;
      int valid = 0;
#pragma unroll 4
      for (int q = 0; q < fp.k; ++q) valid += fp.inv[static_cast<int64_t>(t) * fp.k + q] >= 0;
      int32_t* ctr = fp.fin_ctr + static_cast<int64_t>(t) * nblk + c0 / 16;
      const int old = atomicAdd(ctr, 1);
      if (old == valid - 1) {
        __threadfence();  // acquire the other routes' outputs
        *ctr = 0;         // for a forward that reuses this route layout
        fin_t = t;
      }
    }
    if (fin_t >= 0) finalize_block<DT>(fp, fin_t, c0);
    head += taken;
    __syncwarp();
    if (lane == 0) *fq.head() = head;
    last_progress = global_timer_ns();
  }
}

// Epilogue of a down unit on one finishing warp: expert outputs in the
// activation dtype (one rounding), per-channel scales applied here.
template <int SCALE, int DT, int NB>
__device__ __forceinline__ bool fused_down_epilogue(const FusedParams& fp, const StageHdr& h, int rowA, int rowB,
                                                    int lane, const float (&tot)[4 * NB], const FinQueue& fq,
                                                    FinPending& pend, volatile int* abort_flag) {
  // (fused finalize: rowA = 16 rb + g, so rowA >> 4 is the row block)
  const GemmParams& p = fp.down;
  if (fp.finalize && pend.valid) {
    if (!fin_publish(fp, fq, pend, lane, abort_flag)) return false;
  }
  const int t = lane & 3;
  const int N = p.n_rows;
  const int rows = min(h.rows, kGemvMaxR);
  const int growA = 128 * h.nt + rowA;  // tile rows in order: expert rows 128 nt + 0..127
  const int growB = 128 * h.nt + rowB;
  const bool okA = growA < N, okB = growB < N;
  float scA = 1.0f, scB = 1.0f;
  if (SCALE == SCALE_CHANNEL) {
    if (okA) scA = bf16_bits_to_float(p.scales[static_cast<int64_t>(h.e) * N + growA]);
    if (okB) scB = bf16_bits_to_float(p.scales[static_cast<int64_t>(h.e) * N + growB]);
  }
  const int64_t oc = p.out_cols;
  uint16_t* y = reinterpret_cast<uint16_t*>(p.out) + static_cast<int64_t>(h.m0) * oc;
#pragma unroll
  for (int n = 0; n < NB; ++n) {
    const int rt0 = 8 * n + 2 * t, rt1 = rt0 + 1;
    if (rt0 < rows && okA) y[rt0 * oc + growA] = F16<DT>::from_float(tot[4 * n + 0] * scA);
    if (rt1 < rows && okA) y[rt1 * oc + growA] = F16<DT>::from_float(tot[4 * n + 1] * scA);
    if (rt0 < rows && okB) y[rt0 * oc + growB] = F16<DT>::from_float(tot[4 * n + 2] * scB);
    if (rt1 < rows && okB) y[rt1 * oc + growB] = F16<DT>::from_float(tot[4 * n + 3] * scB);
  }
  if (fp.finalize) {
    // this warp's 16 output columns of the tile's routes: published with the
    // next down unit of this warp (or when it finishes)
    const int c0 = 128 * h.nt + 16 * (rowA >> 4);
    if (c0 < N) pend = FinPending{h.m0, rows, c0, true};
  }
  return true;
}

// Ring walk of one compute group: with two groups the slots of parity grp
// (ring_len even), with one group every slot.
template <int GROUPS>
struct GroupRing {
  int slot;
  uint32_t ph, seq;
  __device__ __forceinline__ void next(int ring_len) {
    slot += GROUPS;
    seq += GROUPS;
    if (slot >= ring_len) {
      slot -= ring_len;
      ph ^= 1u;
    }
  }
};

// This group's stages of one unit (the first already waited for), its share
// of the exchange and, on the finishing group, the epilogue.  One group takes
// every stage of its units: no exchange.
template <int SCALE, int DT, int LAYOUT, int NB, int GROUPS>
__device__ __forceinline__ bool fused_unit(const FusedParams& fp, uint8_t* smem, int stage_bytes, uint64_t* full,
                                           uint64_t* empty, uint64_t* xfull, uint64_t* xempty,
                                           const StageHdr* hdrs, volatile int* abort_flag, float* red,
                                           int ring_len, int grp, int rowA, int rowB, int rb, int lane,
                                           uint32_t ld_row_off, int ld_row7, int ld_chunk, GroupRing<GROUPS>& r,
                                           uint32_t& xj, const FinQueue& fq, FinPending& pend) {
  const StageHdr h = hdrs[r.slot];
  float tot[4 * NB];
#pragma unroll
  for (int j = 0; j < 4 * NB; ++j) tot[j] = 0.0f;
  for (;;) {
    const uint8_t* sA = smem + r.slot * stage_bytes;
    gemv_stage<SCALE, DT, LAYOUT, NB, true>(sA, rowA, rowB, 0, lane, ld_row_off, ld_row7, ld_chunk, tot);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[r.slot]);
    r.next(ring_len);
    if (r.seq > h.last_seq) break;
    if (!warp_wait(&full[r.slot], r.ph, abort_flag, fp.up.err, fp.up.wait_ns)) return false;
  }
  const bool finisher = GROUPS == 1 || static_cast<int>(h.last_seq & 1u) == grp;
  if (GROUPS == 2 && h.last_seq > h.first_seq) {
    // both groups took stages of this unit: meet in exchange buffer xj % 2
    const int b = xj & 1;
    const uint32_t use = xj >> 1;
    ++xj;
    // buffers of the plan's largest NB (bn / 8), so that units of different
    // NB never overlap in them
    float4* rbuf = reinterpret_cast<float4*>(red) + (b * 8 + rb) * (fp.up.bn >> 3) * 32 + lane;
    if (!finisher) {
      if (!warp_wait(&xempty[b], (use & 1u) ^ 1u, abort_flag, fp.up.err, fp.up.wait_ns)) return false;
#pragma unroll
      for (int n = 0; n < NB; ++n)
        rbuf[n * 32] = make_float4(tot[4 * n + 0], tot[4 * n + 1], tot[4 * n + 2], tot[4 * n + 3]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&xfull[b]);
      return true;
    }
    if (!warp_wait(&xfull[b], use & 1u, abort_flag, fp.up.err, fp.up.wait_ns)) return false;
#pragma unroll
    for (int n = 0; n < NB; ++n) {
      const float4 o = rbuf[n * 32];
      tot[4 * n + 0] += o.x;
      tot[4 * n + 1] += o.y;
      tot[4 * n + 2] += o.z;
      tot[4 * n + 3] += o.w;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&xempty[b]);
  } else if (!finisher) {
    return true;
  }
  if (h.type == kItemUp) {
    fused_up_epilogue<SCALE, DT, NB>(fp, h, rowA, rowB, rb, lane, tot);
    return true;
  }
  return fused_down_epilogue<SCALE, DT, NB>(fp, h, rowA, rowB, lane, tot, fq, pend, abort_flag);
}

template <int SCALE, int DT, int LAYOUT, int NBMAX, int GROUPS>
__global__ void __launch_bounds__(fused_threads(GROUPS), GROUPS == 1 ? 2 : 1)
    w4a16_gemv_fused_kernel(const __grid_constant__ FusedParams fp, const __grid_constant__ CUtensorMap tmA1,
                            const __grid_constant__ CUtensorMap tmS1, const __grid_constant__ CUtensorMap tmA2,
                            const __grid_constant__ CUtensorMap tmS2) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const GemmParams& pu = fp.up;
  const int ring_len = pu.stages;  // even with two groups (host)
  const int stage_bytes = pu.stage_bytes;
  uint8_t* ctrl = smem + ring_len * stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl + kFzOffFull);
  uint64_t* empty = reinterpret_cast<uint64_t*>(ctrl + kFzOffEmpty);
  uint64_t* hdrb = reinterpret_cast<uint64_t*>(ctrl + kFzOffHdrBar);
  uint64_t* xfull = reinterpret_cast<uint64_t*>(ctrl + kFzOffXBar);
  uint64_t* xempty = xfull + 2;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + kFzOffFlags);
  volatile int* prod_issued = abort_flag + 1;
  volatile int* prod_stopped = abort_flag + 2;
  StageHdr* hdrs = reinterpret_cast<StageHdr*>(ctrl + kFzOffHdr);
  const FinQueue fq{ctrl};
  float* red = reinterpret_cast<float*>(ctrl + kGemvCtrlBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Two activation warps (even / odd stages) unless the finalize warp is
  // busy; they also issue the group-scale TMA of their stages when both GEMMs
  // load scales by TMA (the producer then issues one TMA per stage).
  const bool two_copy = GROUPS == 2 && !fp.finalize;
  const bool scale_by_copier = two_copy && SCALE == SCALE_GROUP && fp.up.scale_tma && fp.down.scale_tma;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ring_len; ++s) {
      mbar_init(&full[s], 1 + 32);                 // producer (+ TMA bytes), activation lanes
      mbar_init(&empty[s], kGemvComputeWarps / 2);  // the stage's compute group
      mbar_init(&hdrb[s], 1);                       // producer: header written
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&xfull[b], kGemvComputeWarps / 2);
      mbar_init(&xempty[b], kGemvComputeWarps / 2);
    }
    *abort_flag = 0;
    *prod_stopped = 0;
    *fq.tail() = 0;
    *fq.head() = 0;
    *fq.done() = 0;
    for (int i = 0; i < kFinQ; ++i) fq.flag()[i] = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmA2);
  }
  __syncthreads();

  // Everything below reads what route preparation wrote.
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (fp.finalize) {
      // fused finalize: output rows of tokens without a valid route are zero
      // (nothing arrives for them); token t is this CTA's when t % grid == cta
      for (int t = blockIdx.x; t < fp.T; t += gridDim.x) {
        const bool any = __any_sync(0xFFFFFFFFu, lane < fp.k && fp.inv[static_cast<int64_t>(t) * fp.k + lane] >= 0);
        if (any) continue;
        uint4* row = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(fp.out) + static_cast<int64_t>(t) * fp.down.out_cols);
        for (int c = lane; c < fp.down.out_cols / 8; c += 32) row[c] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_s = l2_policy_evict_last();
    // gated gate/up tiles through the 5D whole-tile view (inter a multiple of
    // 64; the host encodes the maps by the same rule)
    const bool gated_up = pu.act == ACT_SWIGLU;
    const bool gate5d = gated_up && (pu.inter % 64) == 0;
    const int n_t = *pu.num_tiles;
    const int nt1 = pu.n_tiles, s1 = pu.splits;
    const GemmParams& pd = fp.down;
    const int nt2 = pd.n_tiles, nch = (nt2 + fp.down_chunk - 1) / fp.down_chunk;
    const int q1 = n_t * nt1 * s1;
    const int qt = q1 + n_t * nch;
    // The producer runs on lane 0 alone (no warp-wide waits or syncs on its
    // issue path, which paces the whole ring) unless group scales of a GEMM
    // have rows that are not 16-byte multiples, whose cp.async pieces take
    // the whole warp.
    const bool solo = SCALE != SCALE_GROUP || (fp.up.scale_tma && fp.down.scale_tma);
    auto produce = [&](auto solo_c) {
    constexpr bool kSolo = decltype(solo_c)::value;
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (kSolo) return mbar_wait(bar, parity, abort_flag, pu.err, pu.wait_ns);
      return warp_wait(bar, parity, abort_flag, pu.err, pu.wait_ns);
    };
    auto wsync = [&]() {
      if (!kSolo) __syncwarp();
    };
    int slot = 0;
    uint32_t ph = 0, seq = 0;
    bool ok = true;
    int q_lane0 = 0;
    if (lane == 0) q_lane0 = atomicAdd(fp.queue, 1);
    // Per-GEMM constants as scalars (a reference chosen at run time between
    // the two parameter blocks would be read through memory at every stage).
    const int n_up = pu.n_rows, n_dn = pd.n_rows, inter = pu.inter;
    const int k_up = pu.K, k_dn = pd.K;
    const bool stma_up = SCALE == SCALE_GROUP && pu.scale_tma, stma_dn = SCALE == SCALE_GROUP && pd.scale_tma;
    const uint16_t* const sc_up = pu.scales;
    const uint16_t* const sc_dn = pd.scales;
    // Issue one stage: header, scales, weights.  One call site, so that the
    // ring state stays in registers.
    auto issue = [&](bool upq, int m, const int4& ti, int nt, int kb, int split, uint32_t first,
                     uint32_t last) -> bool {
      if (!wwait(&empty[slot], ph ^ 1u)) return false;
      uint8_t* sA = smem + slot * stage_bytes;
      uint8_t* sS = sA + kGvOffS;
      const int e = ti.x;
      const int N = upq ? n_up : n_dn;
      // tile rows 0..63 / 64..127: SwiGLU gate rows and their up rows, else consecutive rows
      const int r0 = (upq && gated_up) ? 64 * nt : 128 * nt;
      const int r1 = (upq && gated_up) ? inter + 64 * nt : r0 + 64;
      const CUtensorMap* tmA = upq ? &tmA1 : &tmA2;
      const CUtensorMap* tmS = upq ? &tmS1 : &tmS2;
      const bool stma = upq ? stma_up : stma_dn;
      const bool stma_here = stma && !scale_by_copier;  // else the stage's activation warp issues it
      if (!kSolo && SCALE == SCALE_GROUP && !stma) {
        const int groups_row = (upq ? k_up : k_dn) / kGroup;
        const int g0 = kb * (kGemvBlockK / kGroup);
        const int ng = min(kGemvBlockK / kGroup, groups_row - g0);
        const uint8_t* sbase = reinterpret_cast<const uint8_t*>(upq ? sc_up : sc_dn);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int tr = lane + 32 * j;
          const int grow = tr < 64 ? r0 + tr : r1 + (tr - 64);
          const uint8_t* src = sbase + (static_cast<int64_t>(e) * N + grow) * (groups_row * 2) + g0 * 2;
          copy_scale_piece(sS + tr * kGvScaleRowBytes, src, grow < N ? max(ng, 0) * 2 : 0);
        }
        cp_async_mbar_arrive(&full[slot]);
      }
      if (lane == 0) {
        StageHdr& h = hdrs[slot];
        h.type = upq ? kItemUp : kItemDown;
        h.m = m;
        h.nt = nt;
        h.kb = kb;
        h.e = e;
        h.m0 = ti.y;
        h.rows = ti.z;
        h.split = split;
        h.first_seq = first;
        h.last_seq = last;
      }
      wsync();
      if (lane == 0) {
        mbar_arrive(&hdrb[slot]);
        mbar_arrive_expect_tx(&full[slot], kGvWeightBytes + (stma ? kTileRows * kGvScaleRowBytes : 0));
        if (SCALE == SCALE_GROUP || LAYOUT == LAYOUT_IL) {
          // one box per tile: the weight rows (and their group scales) of the
          // whole 128-row tile -- a 5D view pairs a gated tile's gate and up
          // halves, otherwise the tile's rows are consecutive
          if (upq && gated_up) {
            if (gate5d) {
              tma_load_5d(sA, tmA, &full[slot], kb * (kGemvBlockK / 2), 0, nt, 0, e, pol_w);
              if (stma_here) tma_load_5d(sS, tmS, &full[slot], kb * (kGemvBlockK / kGroup), 0, nt, 0, e, pol_s);
            } else {
              // inter an odd multiple of 32: 64-row boxes of the gate and up halves
              tma_load_3d(sA, tmA, &full[slot], kb * (kGemvBlockK / 2), r0, e, pol_w);
              tma_load_3d(sA + 8192, tmA, &full[slot], kb * (kGemvBlockK / 2), r1, e, pol_w);
              if (stma_here) {
                tma_load_3d(sS, tmS, &full[slot], kb * (kGemvBlockK / kGroup), r0, e, pol_s);
                tma_load_3d(sS + 64 * kGvScaleRowBytes, tmS, &full[slot], kb * (kGemvBlockK / kGroup), r1, e,
                            pol_s);
              }
            }
          } else {
            tma_load_3d(sA, tmA, &full[slot], kb * (kGemvBlockK / 2), r0, e, pol_w);
            if (stma_here) tma_load_3d(sS, tmS, &full[slot], kb * (kGemvBlockK / kGroup), r0, e, pol_s);
          }
        } else {
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
              tma_load_3d(sA + (b * 2 + hh) * 4096, tmA, &full[slot], kb * kGemvBlockK + hh * 128,
                          (b ? r1 : r0) / 2, e, pol_w);
        }
      }
      wsync();
      ++seq;
      if (++slot == ring_len) {
        slot = 0;
        ph ^= 1u;
      }
      return true;
    };
    while (ok) {
      const int q = kSolo ? q_lane0 : __shfl_sync(0xFFFFFFFFu, q_lane0, 0);
      if (q >= qt) break;
      if (lane == 0) q_lane0 = atomicAdd(fp.queue, 1);  // the next entry, taken while this one streams
      // entry -> route tile m, weight tiles [ntb, nte), K blocks [kb0, kb1) of each
      const bool upq = q < q1;
      int m, ntb, nte, kb0, kb1, split;
      if (upq) {
        m = q / (nt1 * s1);
        const int rem = q - m * (nt1 * s1);
        ntb = rem / s1;
        nte = ntb + 1;
        split = rem - ntb * s1;
        kb0 = split * pu.kb_per_split;
        kb1 = min(kb0 + pu.kb_per_split, pu.kb_total);
      } else {
        const int qq = q - q1;
        m = qq / nch;
        const int c = qq - m * nch;
        ntb = c * fp.down_chunk;
        nte = min(ntb + fp.down_chunk, nt2);
        split = 0;
        kb0 = 0;
        kb1 = pd.kb_total;
      }
      const int4 ti = upq ? pu.tiles[m] : pd.tiles[m];
      for (int nt = ntb; nt < nte && ok; ++nt) {
        const uint32_t first = seq, last = seq + static_cast<uint32_t>(kb1 - kb0) - 1u;
        for (int kb = kb0; kb < kb1 && ok; ++kb) ok = issue(upq, m, ti, nt, kb, split, first, last);
      }
    }
    // two end markers, one for each compute group
    for (int j = 0; j < 2 && ok; ++j) {
      if (!wwait(&empty[slot], ph ^ 1u)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        hdrs[slot].type = kItemEnd;
        mbar_arrive(&hdrb[slot]);
        mbar_arrive(&full[slot]);
      }
      wsync();
      ++seq;
      if (++slot == ring_len) {
        slot = 0;
        ph ^= 1u;
      }
    }
    // Wind-down (as in gemv.cuh): publish the stage count for the activation
    // warp, then wait (bounded) for the copies of the last ring of stages.
    if (lane == 0) {
      *prod_issued = static_cast<int>(seq);
      __threadfence_block();
      *prod_stopped = 1;
      volatile int no_abort = 0;
      const uint32_t from = seq > static_cast<uint32_t>(ring_len) ? seq - ring_len : 0;
      for (uint32_t j = from; j < seq; ++j)
        mbar_wait(&full[j % ring_len], (j / ring_len) & 1, &no_abort, pu.err);
    }
    };
    if (solo) {
      if (lane == 0) produce(std::integral_constant<bool, true>());
    } else {
      produce(std::integral_constant<bool, false>());
    }
  } else if (warp == 1 || (GROUPS == 2 && warp == kFinWarp && two_copy)) {
    // ------------------------------------------------------------------ activation rows
    // Two copy warps take the stages of even and odd sequence number: one
    // warp's per-stage work, slowed by the compute warps beside it on its
    // scheduler, would pace the ring together with the producer's.  The
    // fused finalize keeps its warp busy.
    const int cstride = two_copy ? 2 : 1;
    const uint64_t pol_s = l2_policy_evict_last();
    const bool gated_up = pu.act == ACT_SWIGLU;
    const bool gate5d = gated_up && (pu.inter % 64) == 0;
    const int cfirst = warp == 1 ? 0 : 1;
    uint32_t scale_done = static_cast<uint32_t>(cfirst);  // stages below this had their scale TMA issued
    const int need = 8 * pu.n_tiles;  // published row blocks of a finished route tile
    int slot = cfirst, ends = 0;
    uint32_t ph = 0, done = static_cast<uint32_t>(cfirst);
    bool ok = true;
    int src_type = -1, src_m = -1, src = 0, ready_m = -1;
    while (ends < 2 / cstride) {
      if (!warp_wait(&hdrb[slot], ph, abort_flag, pu.err, pu.wait_ns)) {
        ok = false;
        break;
      }
      const StageHdr h = hdrs[slot];
      if (h.type == kItemEnd) {
        if (lane == 0) mbar_arrive_cnt(&full[slot], 32);
        ++ends;
      } else {
        const bool up = h.type == kItemUp;
        if (scale_by_copier) {
          // the stage's group scales (the producer's expect-tx counts them)
          if (lane == 0) {
            uint8_t* sS = smem + slot * stage_bytes + kGvOffS;
            const int c0 = h.kb * (kGemvBlockK / kGroup);
            if (up && gate5d) {
              tma_load_5d(sS, &tmS1, &full[slot], c0, 0, h.nt, 0, h.e, pol_s);
            } else if (up && gated_up) {
              int r0, r1;
              tile_row_bases<GEMM_UP>(pu, h.nt, r0, r1);
              tma_load_3d(sS, &tmS1, &full[slot], c0, r0, h.e, pol_s);
              tma_load_3d(sS + 64 * kGvScaleRowBytes, &tmS1, &full[slot], c0, r1, h.e, pol_s);
            } else {
              int r0, r1;
              if (up) tile_row_bases<GEMM_UP>(pu, h.nt, r0, r1);
              else tile_row_bases<GEMM_DOWN>(fp.down, h.nt, r0, r1);
              tma_load_3d(sS, up ? &tmS1 : &tmS2, &full[slot], c0, r0, h.e, pol_s);
            }
          }
          scale_done = done + cstride;
        }
        const GemmParams& g = up ? fp.up : fp.down;
        const int rows = min(h.rows, kGemvMaxR);
        if (!up && h.m != ready_m) {
          // the intermediate rows of route tile m: wait until every row block
          // of every gate/up weight tile is published
          int rdy = 1;
          if (lane == 0) {
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire_gpu(fp.ready + h.m) < need) {
              if (*abort_flag) {
                rdy = 0;
                break;
              }
              if (global_timer_ns() - t0 > pu.wait_ns) {
                *abort_flag = 1;
                atomicExch(pu.err, kErrTimeout);
                rdy = 0;
                break;
              }
            }
          }
          rdy = __shfl_sync(0xFFFFFFFFu, rdy, 0);
          __syncwarp();  // lane 0's acquire orders the other lanes' copies
          if (!rdy) {
            ok = false;
            break;
          }
          ready_m = h.m;
        }
        if (h.type != src_type || h.m != src_m) {
          src = 0;
          if (lane < rows) {
            if (up) {
              const int route = g.perm[h.m0 + lane];
              src = route >= 0 ? route / g.top_k : 0;
            } else {
              src = h.m0 + lane;
            }
          }
          src_type = h.type;
          src_m = h.m;
        }
        const uint16_t* xsrc = reinterpret_cast<const uint16_t*>(g.x);
        uint8_t* xs = smem + slot * stage_bytes + kGvOffX;
        const int col = h.kb * kGemvBlockK + lane * 8;
        const bool valid = col < g.K;
        for (int r = 0; r < rows; ++r) {
          const int srow = __shfl_sync(0xFFFFFFFFu, src, r);
          cp_async_cg16(xs + r * kGvRouteBytes + lane * 16,
                        xsrc + static_cast<int64_t>(srow) * g.K + (valid ? col : 0), valid ? 16u : 0u);
        }
        cp_async_mbar_arrive_noinc(&full[slot]);
      }
      done += cstride;
      slot += cstride;
      if (slot >= ring_len) {
        slot -= ring_len;
        ph ^= 1u;
      }
    }
    // After an abort: the arrivals owed to this warp's stages that the
    // producer issued beyond its last one (see gemv.cuh).
    if (!ok && lane == 0) {
      const uint64_t t0 = global_timer_ns();
      while (!*prod_stopped && global_timer_ns() - t0 < kWaitTimeoutNs) {
      }
      if (*prod_stopped) {
        __threadfence_block();
        const uint32_t to = static_cast<uint32_t>(*prod_issued);
        for (uint32_t j = done; j < to; j += cstride) {
          mbar_arrive_cnt(&full[j % ring_len], 32);
          // scale bytes the producer counted but this warp never loaded (the
          // slot still holds stage j's header: its reuse needs this arrival)
          if (scale_by_copier && j >= scale_done && hdrs[j % ring_len].type != kItemEnd)
            mbar_complete_tx(&full[j % ring_len], kTileRows * kGvScaleRowBytes);
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp < 2 + 8 * GROUPS) {
    // ------------------------------------------------------------------ compute groups
    const int cw = warp - 2, grp = cw >> 3, rb = cw & 7, g = lane >> 2;
    // rows of this warp: SwiGLU gate/up tiles pair gate row 8 rb + g with its
    // up row; otherwise (ReLU^2 gate/up, down) 16 consecutive rows.  The
    // gate/up row map depends on the activation only, the down tiles always
    // take the plain map: both use tile rows (rowA, rowB) as the stage layout
    // and the epilogues interpret them per GEMM.
    const bool gated = pu.act == ACT_SWIGLU;
    const int rowA_up = gated ? 8 * rb + g : 16 * rb + g;
    const int rowB_up = gated ? 64 + 8 * rb + g : 16 * rb + 8 + g;
    const int rowA_dn = 16 * rb + g, rowB_dn = 16 * rb + 8 + g;
    auto ld_off = [&](int rowA, int rowB, uint32_t& off, int& r7, int& ch) {
      const int ld_i = lane & 7, ld_j = lane >> 3;
      const int ld_row = (ld_j & 1) ? rowB - g + ld_i : rowA - g + ld_i;
      off = (ld_row >> 6) * 8192 + (ld_row & 63) * 128;
      r7 = ld_row & 7;
      ch = ld_j >> 1;
    };
    GroupRing<GROUPS> r;
    r.slot = grp;
    r.ph = 0;
    r.seq = static_cast<uint32_t>(grp);
    uint32_t xj = 0;
    FinPending pend{0, 0, 0, false};
    for (;;) {
      if (!warp_wait(&full[r.slot], r.ph, abort_flag, pu.err, pu.wait_ns)) break;
      const int type = hdrs[r.slot].type;
      if (type == kItemEnd) break;
      const int nb = (min(hdrs[r.slot].rows, kGemvMaxR) + 7) >> 3;
      const bool up = type == kItemUp;
      const int rowA = up ? rowA_up : rowA_dn, rowB = up ? rowB_up : rowB_dn;
      // this lane's ldmatrix row (recomputed per unit: registers are scarce)
      uint32_t off;
      int r7, ch;
      ld_off(rowA, rowB, off, r7, ch);
      bool ok;
#define W4A16_FUSED_UNIT(NBV)                                                                                   \
  fused_unit<SCALE, DT, LAYOUT, NBV, GROUPS>(fp, smem, stage_bytes, full, empty, xfull, xempty, hdrs, abort_flag, red, \
                                     ring_len, grp, rowA, rowB, rb, lane, off, r7, ch, r, xj, fq, pend)
      if (NBMAX == 1 || nb <= 1) ok = W4A16_FUSED_UNIT(1);
      else if (NBMAX == 2 || nb == 2) ok = W4A16_FUSED_UNIT(2);
      else ok = W4A16_FUSED_UNIT(4);
#undef W4A16_FUSED_UNIT
      if (!ok) break;
    }
    if (fp.finalize) {
      // the last down unit's record, then this warp's end
      if (pend.valid && !*abort_flag) fin_publish(fp, fq, pend, lane, abort_flag);
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        atomicAdd(fq.done(), 1);
      }
    }
  } else if (GROUPS == 2) {
    // ------------------------------------------------------------------ finalize
    if (fp.finalize) fin_warp<DT>(fp, fq, lane, abort_flag);
  }
  __syncthreads();
  if (fp.finalize) {
    // The last CTA to finish resets the queue state (no combine launch follows
    // to do it), so that a forward can reuse this route layout.
    __shared__ int last_cta;
    if (threadIdx.x == 0) {
      __threadfence();
      last_cta = atomicAdd(fp.exit_ctr, 1) == static_cast<int>(gridDim.x) - 1;
    }
    __syncthreads();
    if (last_cta) {
      __threadfence();
      for (int i = threadIdx.x; i < fp.reset_len; i += blockDim.x) fp.reset[i] = 0;
    }
  }
}

template <int SCALE, int DT, int LAYOUT, int NBMAX, int GROUPS>
cudaError_t launch_gemv_fused_one(const FusedParams& fp, const CUtensorMap& tmA1, const CUtensorMap& tmS1,
                                  const CUtensorMap& tmA2, const CUtensorMap& tmS2, int grid, int smem_bytes,
                                  cudaStream_t s, bool pdl) {
  auto kern = w4a16_gemv_fused_kernel<SCALE, DT, LAYOUT, NBMAX, GROUPS>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static int configured_for[64] = {0};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured_for[dev] < smem_bytes) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    // two CTAs per SM need the largest shared-memory carveout
    if (e == cudaSuccess && GROUPS == 1)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    configured_for[dev] = smem_bytes;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(fused_threads(GROUPS));
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, fp, tmA1, tmS1, tmA2, tmS2);
}

template <int DT, int LAYOUT>
cudaError_t launch_gemv_fused_dt(int scale_kind, const FusedParams& fp, const CUtensorMap& tmA1,
                                 const CUtensorMap& tmS1, const CUtensorMap& tmA2, const CUtensorMap& tmS2, int grid,
                                 int smem_bytes, cudaStream_t s, bool pdl) {
  // one kernel per largest route block count of the plan's tiles (bn / 8): the
  // 32-route code path costs registers that the 8-route one then lacks
  // (measured: 3-5 % at 1 to 32 tokens on the Kimi shard with 8-route tiles)
#define W4A16_FUSED_ONE(SC, NBM) \
  launch_gemv_fused_one<SC, DT, LAYOUT, NBM, 2>(fp, tmA1, tmS1, tmA2, tmS2, grid, smem_bytes, s, pdl)
  const int bn = fp.up.bn;
  if (fp.groups == 1) {
    // one compute group per CTA, two CTAs per SM
    if (fp.finalize) return cudaErrorInvalidValue;
#define W4A16_FUSED_ONE1(SC, NBM) \
  launch_gemv_fused_one<SC, DT, LAYOUT, NBM, 1>(fp, tmA1, tmS1, tmA2, tmS2, grid, smem_bytes, s, pdl)
    if (scale_kind == SCALE_GROUP)
      return bn <= 8 ? W4A16_FUSED_ONE1(SCALE_GROUP, 1)
                     : (bn <= 16 ? W4A16_FUSED_ONE1(SCALE_GROUP, 2) : W4A16_FUSED_ONE1(SCALE_GROUP, 4));
    return bn <= 8 ? W4A16_FUSED_ONE1(SCALE_CHANNEL, 1)
                   : (bn <= 16 ? W4A16_FUSED_ONE1(SCALE_CHANNEL, 2) : W4A16_FUSED_ONE1(SCALE_CHANNEL, 4));
#undef W4A16_FUSED_ONE1
  }
  if (scale_kind == SCALE_GROUP)
    return bn <= 8 ? W4A16_FUSED_ONE(SCALE_GROUP, 1)
                   : (bn <= 16 ? W4A16_FUSED_ONE(SCALE_GROUP, 2) : W4A16_FUSED_ONE(SCALE_GROUP, 4));
  return bn <= 8 ? W4A16_FUSED_ONE(SCALE_CHANNEL, 1)
                 : (bn <= 16 ? W4A16_FUSED_ONE(SCALE_CHANNEL, 2) : W4A16_FUSED_ONE(SCALE_CHANNEL, 4));
#undef W4A16_FUSED_ONE
}

}  // namespace w4a16
