// Shared definitions of the sm_103a W4A16 MoE kernels: launch parameter
// structs (host <-> device) and thin inline-PTX wrappers for mbarriers, TMA,
// tcgen05 (TMEM allocation, MMA, loads/stores) and programmatic dependent
// launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace w4a16 {

// ---------------------------------------------------------------------------
// Tiling constants
// ---------------------------------------------------------------------------
constexpr int kTileRows = 128;       // weight rows per MMA tile (MMA M)
constexpr int kBlockK = 256;         // K elements per pipeline stage (shared-memory ring)
constexpr int kHalfK = kBlockK / 2;
constexpr int kGroup = 32;           // group size of the group-wise scales
constexpr int kGroupsPerStage = kBlockK / kGroup;
constexpr int kMaxStages = 12;
constexpr int kGemmThreads = 768;    // gate/up GEMM: 24 warps (see the role map in gemm.cuh)
constexpr int kGemmThreadsDown = 896;  // down GEMM: 28 warps, two epilogue warp sets
constexpr int kGemmDqWarps = 16;     // dequantising warps: 4 warpgroups
constexpr int kQuarterK = kBlockK / 4;  // K values each dequant warpgroup handles per stage
constexpr int kTmemCols = 512;
constexpr int kAslotCols = 128;           // one A slot: 16 MMAs (NT tiles x 256/NT K values)
constexpr int kMaxAslots = 3;
constexpr int kMaxNT = 4;                  // weight tiles per tensor-core unit
constexpr int kMaxBN = 128;
// TMEM split: A slots from column 0 (as many 128-column slots as fit, at most
// 3), then acc_bufs accumulator sets of NT tiles x bn columns.
__host__ __device__ constexpr int gemm_a_slots(int nt, int bn, int acc_bufs) {
  return (kTmemCols - acc_bufs * nt * bn) / kAslotCols < kMaxAslots ? (kTmemCols - acc_bufs * nt * bn) / kAslotCols
                                                                     : kMaxAslots;
}
// Tensor-core stage: NT weight tiles (16 KB packed + 2 KB scales each) and the
// route tile's activation rows (bn x 512 B).
__host__ __device__ constexpr int gemm_stage_bytes(int nt, int bn) { return nt * (kTileRows * kBlockK / 2 + kTileRows * 16) + bn * kBlockK * 2; }
constexpr int kStageA = kTileRows * kBlockK / 2;   // 16 KB packed INT4 per stage
constexpr int kStageS = kTileRows * kGroupsPerStage * 2;  // 2 KB BF16 group scales per stage
constexpr int kStageBRow = kBlockK * 2;            // bytes of one activation row per stage
// Down-GEMM output staging: 8 epilogue warps x 2 buffers x 16 routes x 32
// rows of the output element (2 bytes, or 4 for FP32 split partials)
__host__ __device__ constexpr int epi_stage_bytes(bool out16) { return 8 * 2 * 16 * 32 * (out16 ? 2 : 4); }

// CUDA-core GEMV path (gemv.cuh): route tiles of at most kGemvMaxR routes,
// pipeline stages of kGemvBlockK K values; the stage size (and so the number
// of stages) follows the route-tile height, and units of several stages need
// a K-half exchange buffer (ksplit).
constexpr int kGemvThreads = 576;    // 18 warps: see the role map in gemv.cuh
constexpr int kGemvMaxR = 32;
constexpr int kGemvBlockK = 256;
constexpr int kGemvMaxStages = 12;
constexpr int kGemvCtrlBytes = 4608;   // mbarriers, flags, tile table
constexpr int kGemvSmemLimit = 232448;
constexpr int kSmemPerSM = 233472;     // shared memory of one SM (228 KB)
// weights (16 KB) + BF16 scales (2 KB) + rows of bn routes (512 B + 64 B pad each)
__host__ __device__ constexpr int gemv_stage_bytes(int bn) {
  return (kTileRows * kGemvBlockK / 2 + kTileRows * 16 + bn * 576 + 1023) / 1024 * 1024;
}
// control block + two exchange buffers of 8 warps x bn / 8 blocks x 32 lanes x 16 B
__host__ __device__ constexpr int gemv_ctrl_bytes(int bn, bool ksplit) {
  return kGemvCtrlBytes + (ksplit ? 2 * 8 * (bn / 8) * 32 * 16 : 0);
}
__host__ __device__ constexpr int gemv_stages(int bn, bool ksplit) {
  return (kGemvSmemLimit - 1024 - gemv_ctrl_bytes(bn, ksplit)) / gemv_stage_bytes(bn) < kGemvMaxStages
             ? (kGemvSmemLimit - 1024 - gemv_ctrl_bytes(bn, ksplit)) / gemv_stage_bytes(bn)
             : kGemvMaxStages;
}
__host__ __device__ constexpr int gemv_smem_bytes(int bn, bool ksplit) {
  return 1024 + gemv_stages(bn, ksplit) * gemv_stage_bytes(bn) + gemv_ctrl_bytes(bn, ksplit);  // 1 KB slack
}

enum { ACT_SWIGLU = 0, ACT_RELU2 = 1 };
enum { SCALE_GROUP = 0, SCALE_CHANNEL = 1 };
enum { DT_BF16 = 0, DT_FP16 = 1 };
enum { GEMM_UP = 0, GEMM_DOWN = 1 };
// Packed weight layouts.  CANON: the caller's checkpoint layout (group scales:
// two codes per byte along K, even K in the low nibble; per-channel: two rows
// per byte along the output dim).  IL: the plan-time relayout -- always packed
// along K, and inside every 32-bit word (8 consecutive K values 8w..8w+7) the
// nibble at bit position 4p holds K index 8w + {0, 2, 4, 6, 1, 3, 5, 7}[p], so
// that (word >> 4i) & 0x000F000F is the pair (8w + 2i, 8w + 2i + 1).
enum { LAYOUT_CANON = 0, LAYOUT_IL = 1 };

// ---------------------------------------------------------------------------
// Launch parameters
// ---------------------------------------------------------------------------
struct RoutePrepParams {
  const int32_t* ids;      // [T, k]
  int32_t T, k, E, expert_offset, bm;
  int32_t* counts;         // [E]
  int32_t* offs;           // [E + 1]
  int32_t* perm;           // [slots_cap]
  int32_t* inv;            // [T * k]
  int4* tiles;             // [tiles_cap]
  int32_t* num_tiles;      // [1]
  int32_t* counters;       // [ctr_len] split-K arrival counters, zeroed here
  int32_t ctr_len;
  int32_t* err;            // device error flag, cleared here
  int32_t* cta_hist;       // [n_cta][E] expert counts of each CTA's routes (n_cta > 1)
  int32_t n_cta, tpc;      // CTAs and whole tokens per CTA (the last CTA may get fewer)
  // router front end (logits != NULL): softmax + top-k over G experts writes
  // ids_out / weights_out [T, k], which the placement then reads as `ids`
  const float* logits;
  int32_t G;
  int32_t* ids_out;
  float* weights_out;
};
// Route preparation: at most kRouteMaxCtas CTAs (the expert totals are summed
// over them by every CTA of the placement kernel).
constexpr int kRouteMaxCtas = 64;

struct GemmParams {
  int32_t act;             // ACT_* (gate/up GEMM epilogue)
  int32_t E;               // local experts
  int32_t n_rows;          // weight rows per expert: N1 (gate/up) or H (down)
  int32_t K;               // reduction length: H (gate/up) or I (down)
  int32_t inter;           // I
  int32_t out_cols;        // row length of the output buffer (I or H)
  int32_t bn;              // route-tile height = MMA N
  int32_t n_tiles;         // 128-row weight tiles per expert
  int32_t nt_unit;         // tensor-core path: weight tiles per unit (NT = 1, 2, 4)
  int32_t n_groups;        // tensor-core path: ceil(n_tiles / NT) unit groups per route tile
  int32_t acc_bufs;        // tensor-core path: accumulator sets in TMEM (1 or 2)
  int32_t kb_total;        // K blocks of kBlockK
  int32_t splits;          // split-K factor
  int32_t kb_per_split;
  int32_t tail_max;        // tensor-core gate/up without split-K: at most this many K pieces
                           // for each unit of the last, partial wave (0 or 1: none)
  int32_t stages;
  int32_t top_k;
  int32_t stage_bytes;
  const int4* tiles;       // route tiles (expert, first slot, valid rows, 0)
  const int32_t* num_tiles;
  const int32_t* perm;     // slot -> flat route (gate/up: activation rows by token)
  const void* x;           // gate/up: activations [T, H] (both paths); down, CUDA-core
                           // path: the intermediate [slots_cap, I]
  const uint16_t* scales;  // BF16 scale bits of this GEMM's weights
  int64_t slots_cap;
  void* out;               // gate/up: intermediate [slots_cap, I] act dtype
                           // down: FP32 partial outputs [splits, slots_cap, H]
  float* part;             // gate/up split-K partials [splits, slots_cap, N1]; with tail
                           // pieces instead [pieces, NT, bn, 128] (piece-major, then tile,
                           // route, TMEM lane)
  int32_t* counters;       // gate/up split-K arrival counters [tiles_cap * n_tiles]
  int32_t* err;
  int32_t tiles_cap;       // capacity of `tiles`
  int32_t scale_tma;       // group scales loaded by TMA (their rows are 16-byte multiples)
  int32_t out16;           // down GEMM: expert outputs in the activation dtype (no split-K),
                           // else FP32 split partials
  int32_t masked_rows;     // down GEMM, masked-count layout: the output is [E][masked_rows][H]
                           // (expert e's slot offs[e] + i to row i; rows past max are dropped)
  const int32_t* seg_offs; // ... with the experts' first slots (route preparation's offsets)
  uint64_t wait_ns;        // limit of every pipeline wait (drains use kWaitTimeoutNs)
};

// Both CUDA-core GEMMs in one launch (gemv_fused.cuh).
constexpr int kMaxFusedSplits = 8;  // gate/up split-K factor of the fused launch
struct FusedParams {
  GemmParams up;           // gate/up GEMM: x -> intermediate (split-K partials in up.part)
  GemmParams down;         // down GEMM: intermediate -> expert outputs y (activation dtype)
  int32_t* queue;          // [1] work-queue head, zeroed by route preparation
  int32_t* ready;          // [tiles_cap] published gate/up row blocks per route tile
  int32_t* fix;            // [tiles_cap * nt1 * 8] split arrivals per (route tile, weight tile, row block)
  int32_t down_chunk;      // down weight tiles per queue entry
  // Fused finalize (finalize != 0): the down epilogue combines the expert
  // outputs itself (no combine launch).  Per (token, 16-column block) arrival
  // counters elect the last route's warp, which sums the token's routes in
  // top-k order with the combine's arithmetic; the last CTA to exit resets the
  // queue state.
  int32_t finalize;
  int32_t* fin_ctr;        // [T * H / 16]
  const int32_t* inv;      // [T * k] slot of each route, -1 when invalid
  const float* topk_weights;
  int32_t T, k, renormalize;
  void* out;               // [T, H] act dtype
  int32_t* exit_ctr;       // CTAs done (inside the reset range)
  int32_t* reset;          // [reset_len] queue state zeroed by the last CTA
  int32_t reset_len;
  int32_t groups;          // compute groups per CTA: 2 (one CTA per SM) or 1 (two CTAs per SM,
                           // no fused finalize)
};

struct CombineParams {
  const void* y;           // [splits, slots_cap, H]: activation dtype when y16, else FP32
  int32_t y16;
  int64_t slots_cap;
  int32_t splits;
  const int32_t* inv;      // [T * k]
  const float* topk_weights;
  int32_t T, H, k, renormalize;
  void* out;               // [T, H] act dtype
  int32_t* zero;           // counters to reset once the expert GEMMs are done (or NULL)
  int32_t zero_len;
};

// Host-side launchers (one translation unit each).
cudaError_t launch_route_prep(const RoutePrepParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_gemm(int which, int scale_kind, int dtype, int layout, const GemmParams& p,
                        const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                        const CUtensorMap& tmS, int grid, int smem_bytes, cudaStream_t s, bool pdl);
cudaError_t launch_gemv(int which, int scale_kind, int dtype, int layout, const GemmParams& p,
                        const CUtensorMap& tmA, const CUtensorMap& tmS, int grid, int smem_bytes,
                        cudaStream_t s, bool pdl);
cudaError_t launch_gemv_fused(int scale_kind, int dtype, int layout, const FusedParams& p, const CUtensorMap& tmA1,
                              const CUtensorMap& tmS1, const CUtensorMap& tmA2, const CUtensorMap& tmS2, int grid,
                              int smem_bytes, cudaStream_t s, bool pdl);
cudaError_t launch_combine(int dtype, const CombineParams& p, cudaStream_t s, bool pdl);
// Checkpoint layout -> LAYOUT_IL for one packed weight tensor of E experts x N
// rows x K values (row_pairs: per-channel [E, N/2, K] input, else [E, N, K/2]).
cudaError_t launch_relayout(bool row_pairs, const uint8_t* in, uint8_t* out, int64_t E, int32_t N, int32_t K,
                            int num_sms, cudaStream_t s);

constexpr int kRoutePrepThreads = 1024;
constexpr int kRoutePrepWarps = kRoutePrepThreads / 32;

#if defined(__CUDACC__)

// Error codes written to the device error flag.
constexpr int kErrTimeout = 1;
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s: default and drain limit

// ---------------------------------------------------------------------------
// Generic helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}


// Programmatic dependent launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

// Transaction bytes counted as arrived without a copy (abort paths: bytes
// of copies that will never be issued).
__device__ __forceinline__ void mbar_complete_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// `count` arrivals at once.
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t count) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)), "r"(count)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase (mbarrier.try_wait may instead suspend the
// thread in hardware until the phase completes or a system-defined time
// passes).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: returns false when the CTA-wide abort flag is raised or the
// wait has lasted `limit_ns`, after raising the abort flag and the global
// error flag.  Every spin in the GEMM pipelines goes through here: pipeline
// waits pass the plan's limit (GemmParams::wait_ns), the waits that drain
// copies and MMAs still in flight before a CTA exits pass kWaitTimeoutNs.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                   int32_t* err, uint64_t limit_ns) {
  // Checked after every attempt.  Limits shorter than the default poll with
  // test_wait (a try_wait can outlast them while suspended), so a limit of one
  // timer tick gives up after one tick.
  const bool poll = limit_ns < kWaitTimeoutNs;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicExch(err, kErrTimeout);
      return false;
    }
  }
}

// Fast path inline (one try_wait), the bounded spin out of line: the wait is
// used at many sites and inlining the spin loop everywhere bloats the code
// that all warp roles share in the instruction cache.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                          uint64_t limit_ns = kWaitTimeoutNs) {
  if (limit_ns < kWaitTimeoutNs ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, err, limit_ns);
}

// One lane of a converged warp, chosen by the hardware (elect.sync).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t"
      "elect.sync _|P1, 0xffffffff;\n\t"
      "selp.b32 %0, 1, 0, P1;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Next use of a ring of `stages` slots: slot index and the parity of its phase.
__device__ __forceinline__ void ring_next(int& st, uint32_t& ph, int stages) {
  if (++st == stages) {
    st = 0;
    ph ^= 1u;
  }
}

// ---------------------------------------------------------------------------
// TMA (tensor) loads, completion signalled on an mbarrier as transaction bytes
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
      "cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2, int c3, int c4, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
      "cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
      "cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

// Store a box of a 2D tensor from shared memory; completion is tracked by the
// issuing thread's bulk async-groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until all of this thread's bulk groups have completed (writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Ampere-style asynchronous copies (used for the small group-scale tiles whose
// global row stride is not a multiple of 16 bytes in general).
template <int BYTES>
__device__ __forceinline__ void cp_async(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(smem_u32(dst)), "l"(src),
               "n"(BYTES)
               : "memory");
}

// The BF16 group scales of one row for one stage: nbytes (even, <= 16) from
// global src into the 16-byte shared slot dst, the rest zeroed.  One 16-byte
// cp.async when the piece is whole and 16-byte aligned, 4-byte cp.async
// pieces when it is 4-byte aligned, else 16-bit loads and stores (rows of an
// odd number of groups -- K an odd multiple of 32 -- are only 2-byte
// aligned).  The caller then arrives on the stage barrier with
// cp.async.mbarrier.arrive (which waits for the copies) and, after a
// __syncwarp, publishes the plain stores through one lane's release arrive.
__device__ __forceinline__ void copy_scale_piece(uint8_t* dst, const uint8_t* src, int nbytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(src);
  if (nbytes == 16 && (a & 15) == 0) {
    cp_async<16>(dst, src);
    return;
  }
  if ((a & 3) == 0 && (nbytes & 3) == 0) {
    for (int o = 0; o < nbytes; o += 4) cp_async<4>(dst + o, src + o);
  } else {
    for (int o = 0; o < nbytes; o += 2)
      *reinterpret_cast<uint16_t*>(dst + o) = *reinterpret_cast<const uint16_t*>(src + o);
  }
  for (int o = nbytes; o < 16; o += 2) *reinterpret_cast<uint16_t*>(dst + o) = 0;
}

// 16-byte copy that bypasses L1; copies src_bytes (0 or 16) and zero-fills the rest.
__device__ __forceinline__ void cp_async_cg16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}

// Arrive on `bar` once this thread's earlier cp.async copies have landed; the
// barrier's expected count includes this arrival (no pending-count increment).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive on `bar` once this thread's earlier cp.async copies have landed; the
// pending count is raised first, so the barrier's expected count is unchanged.
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, loads and stores
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] x B[smem]^T, kind::f16 (BF16/FP16 in, FP32 accumulate).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same MMA with the B descriptor given as two 32-bit halves (the address
// fields live in the low half; offsets added there never reach the high half).
__device__ __forceinline__ void mma_ts_lh(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 bd;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "mov.b64 bd, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Instruction descriptor of kind::f16: FP32 accumulator, A and B of the same
// 16-bit type (bf16 when `bf16`), both K-major, shape M x N.
__host__ __device__ constexpr uint32_t make_idesc_f16(bool bf16, int m, int n) {
  return (1u << 4)                                   // D format: F32
         | ((bf16 ? 1u : 0u) << 7)                   // A format
         | ((bf16 ? 1u : 0u) << 10)                  // B format
         | (static_cast<uint32_t>(n >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24);    // M / 16
}

// Shared-memory matrix descriptor: K-major operand stored with the 128-byte
// swizzle (rows of 128 bytes, 8-row atoms of 1024 bytes).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);          // start address
  d |= static_cast<uint64_t>(1) << 16;                        // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                // stride byte offset: 8 rows
  d |= static_cast<uint64_t>(1) << 46;                        // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                        // swizzle: 128B
  return d;
}

// 32 lanes x 32 bit, repeated over N consecutive columns.  No "memory" clobber:
// the stores only read registers; tcgen05.wait::st (which has one) orders them.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]));
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Waits for this thread's TMEM loads with their 16 destination registers as
// in/out operands, so that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(float (&v)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]), "+f"(v[7]),
                 "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]), "+f"(v[14]),
                 "+f"(v[15])
               :
               : "memory");
}

__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) ^ c
  return d;
}

#endif  // __CUDACC__

}  // namespace w4a16
