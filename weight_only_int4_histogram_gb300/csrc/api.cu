// Host side of the C ABI in include/w4a16_moe.h: descriptor validation, the
// per-batch planner (GEMM path, route-tile height, split-K factors,
// persistent grid sizes, workspace layout), TMA descriptor encoding and the
// launch sequence
//   route_prep -> gate/up GEMM -> down GEMM -> combine
// chained with programmatic dependent launch; the plan-time weight relayout.  Both GEMMs run either on the
// tensor cores (gemm.cuh) or, when experts see only a few routes each, on the
// CUDA cores (gemv.cuh).  No allocation, host sync or
// device->host copy happens in prepare_routes / forward.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "common.cuh"
#include "masked.cuh"
#include "router.cuh"
#include "w4a16_moe.h"

using namespace w4a16;

struct w4a16_moe_plan_s {
  w4a16_moe_desc d;
  int num_sms;
  int ov_bn, ov_s1, ov_s2;
  int ov_nt1, ov_nt2;  // tuning: weight tiles per tensor-core unit (0 = automatic)
  int path;    // W4A16_PATH_*
  int layout;  // W4A16_LAYOUT_* of the weights later forwards receive
  uint64_t wait_ns;  // limit of the GEMM pipelines' bounded waits
  size_t ws_bytes;
  bool pdl;
  bool fused;        // CUDA-core path: both GEMMs in one launch
  bool finalize;     // fused launch: combine inside the down epilogue (no combine launch)
  int ov_chunk;      // tuning: down weight tiles per fused queue entry (0 = automatic)
  int tail_max;      // tensor-core gate/up: K pieces per unit of the last partial wave (<= 1: none)
  int ov_stages;     // tuning: tensor-core ring stages at most (0 = as many as fit)
  int ov_bn_cc;      // tuning: CUDA-core route-tile height (8, 16, 32; 0 = automatic)
  int ov_fgroups;    // tuning: fused launch compute groups per CTA (1, 2; 0 = automatic)
  cudaEvent_t ev[4];
  bool has_ev;
};

namespace {

thread_local std::string g_err;

w4a16_status fail(w4a16_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

w4a16_status cuda_fail(cudaError_t e, const char* what) {
  return fail(W4A16_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int cdiv(int a, int b) { return (a + b - 1) / b; }

struct Layout {
  bool gemv;  // CUDA-core path for both GEMMs
  bool fused;       // CUDA-core path: both GEMMs in one launch (gemv_fused.cuh)
  int fgroups;      // fused: compute groups per CTA (2: one CTA per SM; 1: two CTAs per SM)
  int down_chunk;   // fused: down weight tiles per queue entry
  int ctr_len;      // counters zeroed by route preparation
  bool fin;         // fused finalize in this forward
  int tail;         // tensor-core gate/up: tail pieces per unit at most (0: none)
  int fix_len;      // fused: queue head + ready counts + split counters (reset after a forward)
  int T, R, bn, tiles_cap;
  int64_t slots_cap;
  int n1;
  int nt1, kb1, s1, kbps1;
  int nt2, kb2, s2, kbps2;
  int ntu1, ntu2;          // tensor-core path: weight tiles per unit (NT) of each GEMM
  int acc1, acc2;          // tensor-core path: accumulator sets in TMEM
  int stage_bytes2;        // tensor-core down GEMM stage
  int stages, stage_bytes, smem;   // gate/up GEMM (and the CUDA-core path's both GEMMs)
  int stages2, smem2;              // tensor-core down GEMM (output staging buffers)
  int grid1, grid2;
  size_t off_err, off_counts, off_offs, off_ntiles, off_tiles, off_perm, off_inv, off_ctr, off_chist;
  size_t off_part, off_inter, off_y;
  size_t off_sx, off_sids, off_sw, off_sout;  // host-call staging (w4a16_moe_forward_host / masked)
  size_t total;
};

// Expected routes per local expert up to which the warp-MMA GEMV runs both
// GEMMs; above it the tcgen05 path wins (its MMA time per weight is the same
// for any tile fill up to 64 routes).  Measured crossovers on GB300 (whole
// forward, both paths forced, graph replay): group scales -- the Kimi shape
// (E 384, H 7168, I 256) is faster on CUDA cores at 10.7 routes per expert
// (357 vs 380 us), even at 12 (384 vs 388) and slower at 13.3 (409 vs 388);
// the 32-of-256-expert shard (H 7168, I 2048) faster at 10 (212 vs 239) and
// slower at 12 (247 vs 236).  Per-channel scales -- E 60, H 2048, I 1408 is
// faster on CUDA cores through 30 routes per expert (125 vs 138 us at 21,
// 147 vs 153 at 30); the skewed ReLU^2 E 64, H 2688, I 1856 at 18 (148 vs
// 172) but not at 24 (166 vs 163).  When both GEMMs reduce over at least
// 2048 values (every GEMV unit streams eight or more 256-value stages) the
// GEMV stays ahead much longer: on the 32-expert H = 7168, I = 2048 shape it
// was faster through 64 routes per expert and slower at 96.
constexpr double kGemvMaxRoutesGroup = 11.0;
constexpr double kGemvMaxRoutesChannel = 24.0;
constexpr double kGemvMaxRoutesLongK = 80.0;

// Expected routes per local expert of a T-token batch under uniform routing
// over the declared global experts (the local count when none is declared).
double routes_per_expert(const w4a16_moe_plan_s& P, int T) {
  const int eg = P.d.global_experts > 0 ? P.d.global_experts : P.d.num_experts;
  return static_cast<double>(T) * P.d.top_k / eg;
}

bool use_gemv(const w4a16_moe_plan_s& P, int T) {
  if (P.path == W4A16_PATH_TENSOR_CORES) return false;
  if (P.path == W4A16_PATH_CUDA_CORES) return true;
  const double lam = routes_per_expert(P, T);
  // Without a declared global expert count an expert-parallel shard's
  // routing density is overestimated by global / local; the long-K limit
  // below was measured that way (8 x on the 32-of-256-expert shape).
  const bool long_k = P.d.global_experts == 0 && P.d.hidden >= 2048 && P.d.inter >= 2048;
  const double limit = long_k ? kGemvMaxRoutesLongK
                              : (P.d.scale_kind == W4A16_SCALE_GROUP32_K ? kGemvMaxRoutesGroup
                                                                        : kGemvMaxRoutesChannel);
  return lam <= limit;
}

// CUDA-core path: route tiles of 8, 16 or 32 routes (one, two or four MMA N
// blocks).  Taller tiles stream an expert's weights fewer times but take
// larger stages (a shallower ring); measured on GB300 they pay off from about
// 4 (16 routes) and 10 (32 routes) expected routes per expert.
int choose_bn_gemv(const w4a16_moe_plan_s& P, int T) {
  if (P.ov_bn_cc == 8 || P.ov_bn_cc == 16 || P.ov_bn_cc == kGemvMaxR) return P.ov_bn_cc;
  const double lam = routes_per_expert(P, T);
  return lam <= 4.0 ? 8 : (lam <= 10.0 ? 16 : kGemvMaxR);
}

constexpr int kAutoMaxBN = 64;

// Tensor-core path: weight tiles per unit.  The NT tiles of a unit share each
// stage's activation tile, so the activation rows cross from L2 into shared
// memory once per NT tiles instead of once per tile (at 64-route tiles one
// tile's activation stage is twice its weight stage).  The largest NT in
// {max_nt, ..., 2, 1} that is still needed for the expert's tile count, leaves
// room for 2 stages in the ring and 2 A slots in TMEM -- with two accumulator
// sets when `double_acc` (units of few K blocks, where the epilogue must
// overlap the next unit's MMAs), else with one if two do not fit.
void choose_nt(int n_tiles, int bn, int smem_budget, int max_nt, bool double_acc, int& nt, int& acc_bufs) {
  (void)double_acc;
  // two accumulator sets whenever they fit (measured: the epilogue overlap
  // they give outweighs a third A slot even for 28-stage units)
  for (int acc = 2; acc >= 1; --acc) {
    nt = max_nt;
    while (nt > 1 && (nt / 2 >= n_tiles || smem_budget / gemm_stage_bytes(nt, bn) < 2 ||
                      gemm_a_slots(nt, bn, acc) < 2))
      nt >>= 1;
    acc_bufs = acc;
    if (smem_budget / gemm_stage_bytes(nt, bn) >= 2 && gemm_a_slots(nt, bn, acc) >= 2) return;
  }
}

// Fused CUDA-core launch: one compute group per CTA and two CTAs per SM
// (rings of 4 / 3 / 2 stages at 8 / 16 / 32-route tiles; each group owns
// whole units and its own ring, so one group's
// epilogue never holds up the other's stages) once the expected gate/up units
// fill this many waves of those CTAs; with fewer units, two groups splitting
// each unit's stages finish the gate/up phase sooner.  Measured (whole
// forward, one group vs two): Kimi shard 24 / 32 / 64 tokens (1.99 / 2.46 /
// 3.7 waves) 120.5 / 138.9 / 200.4 vs 126.6 / 147.1 / 212.6 us, but 8 / 16
// tokens (0.78 / 1.43) 70.3 / 104.1 vs 63.1 / 99.0; DeepSeek-like 32-of-256
// shard 32 / 64 tokens (2.13 / 2.9) 131.7 / 163.5 vs 134.8 / 173.7; ReLU^2
// E64 32 tokens (2.96) 85.6 vs 91.8 but 8 tokens (1.67) 50.8 vs 44.7;
// per-channel E60 16 / 32 tokens (2.85 / 3.8) 55.9 / 69.3 vs 59.0 / 73.4.
// Taller tiles: Kimi shard 256 / 384 tokens 284.3 / 306.7 vs 296.6 / 319.1,
// ReLU^2 E64 64 / 128 tokens 106.6 / 128.7 vs 114.3 / 138.9.
constexpr double kOneGroupWaves = 1.9;
// Ring stages of one CTA of the one-group form: half the SM's shared memory
// less the CTA's 1 KB reserve, the alignment slack and the control block.
int gemv_stages1(int bn) {
  return std::min(kGemvMaxStages, (kSmemPerSM / 2 - 1024 - 1024 - kGemvCtrlBytes) / gemv_stage_bytes(bn));
}

// Units of at most this many K blocks keep two accumulator sets.
constexpr int kDoubleAccMaxKb = 8;
// Default weight tiles per tensor-core unit.  Measured on the 384-expert
// H 7168 / I 256 shape at 1024 and 2048 tokens: 2 tiles per unit beat 1 (the
// activation stage crosses from L2 half as often) and 4 (only two 106 KB
// stages fit in shared memory, and units four times larger leave more of
// the last wave idle).
constexpr int kDefaultNT = 2;

// Tensor-core gate/up GEMM: units of the last, partial wave are cut into at
// most this many K pieces (summed by the last piece in piece order), so that
// the wave's few units do not keep most SMs idle for a whole unit.  Measured
// on the Kimi shard (768 units on 152 SMs): 1024 / 2048 tokens 427.7 / 504.5 us
// uncut, 422.6 / 498.3 with 2 pieces, 422.5 / 501.3 with 4, 432.8 / 513.6 with
// 8 -- the few units of a last wave run faster than a full wave's (they have
// the memory system to themselves), so the gain is small.
constexpr int kDefaultTailPieces = 2;

int choose_bn(const w4a16_moe_plan_s& P, int T) {
  if (P.ov_bn) return P.ov_bn;
  // Route-count-based tile height: expected routes per expert plus three
  // standard deviations, so that one route tile usually covers an expert
  // (every extra tile of an expert streams its weights once more), at most
  // kAutoMaxBN = 64 routes.  A stage holds the tile's activation rows (512
  // bytes each): above 64 routes only one weight tile per unit fits, the
  // activation rows then cross from L2 once per weight tile, and on GB300
  // that cost more than the second weight pass it saves (measured at 2048
  // tokens on the 32-local-expert H 7168 / I 2048 shape and at 4096 on the
  // skewed ReLU^2 shape; only the 60-expert per-channel shape at 1024 tokens
  // gained).
  const double lam = routes_per_expert(P, T);
  const double want = lam + 3.0 * std::sqrt(lam) + 1.0;
  int bn = static_cast<int>(std::ceil(want / 16.0)) * 16;
  // Exception: short gate/up reductions (at most 8 stages of 256) whose
  // experts a 96-route tile covers where 64 would take two tiles: one tile
  // per expert dequantises every weight once instead of twice, which outweighs
  // the shallower ring on such short units (the 60-expert H 2048 per-channel
  // shape at 1024 tokens: 239 -> 186 us; the long-K shapes got slower).
  if (bn > kAutoMaxBN && bn <= 96 && cdiv(P.d.hidden, kBlockK) <= 8) return 96;
  return std::min(kAutoMaxBN, std::max(16, bn));
}

// Gate/up split-K factor of the fused CUDA-core launch: the smallest that
// gives every SM a gate/up queue entry (the down entries wait for the gate/up
// rows of their route tile, so SMs without gate/up work would idle until the
// first route tiles are done), at most kMaxFusedSplits.
int choose_fused_splits(double tiles_est, int nt1, int kb, int num_sms) {
  int best = 1;
  for (int s = 1; s <= std::min(kb, kMaxFusedSplits); ++s) {
    if (cdiv(kb, cdiv(kb, s)) != s) continue;
    best = s;
    if (tiles_est * nt1 * s >= num_sms) break;
  }
  return best;
}

// Split-K factor for the expected number of route tiles.  With at least one
// full wave of units, none: every split writes FP32 partials that the last
// one reads back, which costs far more than the wave quantisation it removes
// (the Kimi shard at 2048 tokens, 768 units on 152 SMs: 2 splits 1233 us, none
// 501; the gate/up GEMM's partial last wave is cut into K pieces instead).
// Below one wave the cost model is (waves of units) x (K blocks per unit +
// per-unit overhead); among factors within 5% of the cheapest, the smallest
// wins.
int choose_splits(double tiles_est, int n_tiles, int kb, int num_sms, double overhead) {
  if (tiles_est * n_tiles >= num_sms) return 1;
  double cost[65] = {0};
  double best_cost = 1e300;
  const int smax = std::min(kb, 64);
  for (int s = 1; s <= smax; ++s) {
    const int kbps = cdiv(kb, s);
    cost[s] = 1e300;
    if (cdiv(kb, kbps) != s) continue;
    const double units = tiles_est * n_tiles * s;
    const double waves = std::ceil(units / num_sms);
    cost[s] = waves * (kbps + overhead);
    best_cost = std::min(best_cost, cost[s]);
  }
  for (int s = 1; s <= smax; ++s)
    if (cost[s] <= best_cost * 1.05) return s;
  return 1;
}

Layout make_layout(const w4a16_moe_plan_s& P, int T) {
  const w4a16_moe_desc& d = P.d;
  Layout L = {};
  L.T = T;
  L.R = T * d.top_k;
  L.gemv = use_gemv(P, T);
  L.bn = L.gemv ? choose_bn_gemv(P, T) : choose_bn(P, T);
  const int E = d.num_experts;
  const int touched_max = std::min(E, std::max(L.R, 1));
  L.tiles_cap = (L.R + touched_max * (L.bn - 1)) / L.bn + 1;
  L.slots_cap = static_cast<int64_t>(L.R) + static_cast<int64_t>(touched_max) * (L.bn - 1) + L.bn;
  const bool gated = d.act == W4A16_ACT_SWIGLU;
  L.n1 = gated ? 2 * d.inter : d.inter;
  // SwiGLU tiles pair 64 gate rows with their 64 up rows (the last tile of an
  // inter that is an odd multiple of 32 is half used)
  L.nt1 = gated ? cdiv(d.inter, 64) : cdiv(d.inter, kTileRows);
  const int block_k = L.gemv ? kGemvBlockK : kBlockK;  // K values per pipeline stage
  L.kb1 = cdiv(d.hidden, block_k);
  L.nt2 = cdiv(d.hidden, kTileRows);
  L.kb2 = cdiv(d.inter, block_k);
  // expected route tiles (uniform routing over the declared global experts):
  // touched local experts x tiles per expert
  const double r_loc = routes_per_expert(P, T) * E;  // expected local routes
  const double touched = std::max(1.0, E * (1.0 - std::exp(-r_loc / E)));
  const double per = r_loc / touched;
  const double tiles_est = touched * std::max(1.0, std::ceil(per / L.bn));
  // unit groups per route tile on the tensor-core path (NT tiles per unit; the
  // same choice choose_nt makes below for a full-size ring)
  int g1 = L.nt1, g2 = L.nt2;
  if (!L.gemv) {
    int nt, ab;
    choose_nt(L.nt1, L.bn, 232448 - 3072, P.ov_nt1 ? P.ov_nt1 : kDefaultNT, L.kb1 <= kDoubleAccMaxKb, nt, ab);
    g1 = cdiv(L.nt1, nt);
    choose_nt(L.nt2, L.bn, 232448 - 3072 - epi_stage_bytes(false), P.ov_nt2 ? P.ov_nt2 : kDefaultNT, L.kb2 <= kDoubleAccMaxKb,
              nt, ab);
    g2 = cdiv(L.nt2, nt);
  }
  L.fused = L.gemv && P.fused;
  L.fgroups = 2;
  if (L.fused && !P.finalize && gemv_stages1(L.bn) >= 2 &&
      (P.ov_fgroups == 1 || (P.ov_fgroups == 0 && tiles_est * L.nt1 >= kOneGroupWaves * 2 * P.num_sms)))
    L.fgroups = 1;
  if (L.fused) {
    const int ctas = P.num_sms * (L.fgroups == 1 ? 2 : 1);
    L.s1 = P.ov_s1 ? std::min(P.ov_s1, kMaxFusedSplits) : choose_fused_splits(tiles_est, L.nt1, L.kb1, ctas);
    // every split must own K blocks: each one's arrival completes its row blocks
    L.s1 = cdiv(L.kb1, cdiv(L.kb1, L.s1));
    L.s2 = 1;  // the down GEMM is balanced by the queue instead
    // down weight tiles per queue entry (single-stage down units): 4 with two
    // compute groups per CTA, 2 with one (Kimi shard 32 / 256 tokens 137.9 /
    // 282.3 us against 139.9 / 284.3 with 4 and 143.0 / 288.4 with 8)
    L.down_chunk = P.ov_chunk > 0 ? P.ov_chunk : (L.kb2 == 1 ? (L.fgroups == 1 ? 2 : 4) : 1);
  } else {
    L.s1 = P.ov_s1 ? P.ov_s1 : choose_splits(tiles_est, g1, L.kb1, P.num_sms, 1.5);
    L.s2 = P.ov_s2 ? P.ov_s2 : choose_splits(tiles_est, g2, L.kb2, P.num_sms, 1.0);
  }
  L.kbps1 = cdiv(L.kb1, L.s1);
  L.kbps2 = cdiv(L.kb2, L.s2);
  if (L.gemv) {
    // K-half exchange buffers unless both GEMMs have single-stage units only
    const bool ksplit = L.fused || !(L.kb1 == 1 && L.s1 == 1 && L.kb2 == 1 && L.s2 == 1);
    L.stage_bytes = gemv_stage_bytes(L.bn);
    L.stages = gemv_stages(L.bn, ksplit);
    L.smem = gemv_smem_bytes(L.bn, ksplit);
    if (L.fgroups == 1) {
      // one compute group per CTA (no exchange buffers), two CTAs per SM:
      // each CTA gets half of the SM's shared memory less its 1 KB reserve
      L.stages = gemv_stages1(L.bn);
      L.smem = 1024 + L.stages * L.stage_bytes + kGemvCtrlBytes;
    } else if (L.fused) {
      // the two compute groups take the stages of their parity: an even ring
      L.stages &= ~1;
      L.smem = 1024 + L.stages * L.stage_bytes + gemv_ctrl_bytes(L.bn, true);
    }
    L.stages2 = L.stages;
    L.smem2 = L.smem;
    L.ntu1 = L.ntu2 = 1;
    L.acc1 = L.acc2 = 2;
  } else {
    // dynamic shared memory: 1 KB alignment slack + stages + 2 KB control block
    // (mbarriers, TMEM address, flags)
    const int smem_budget = 232448 - 3072;
    choose_nt(L.nt1, L.bn, smem_budget, P.ov_nt1 ? P.ov_nt1 : kDefaultNT, L.kbps1 <= kDoubleAccMaxKb, L.ntu1, L.acc1);
    const int epi_bytes = epi_stage_bytes(L.s2 == 1);  // 16-bit expert outputs unless split
    choose_nt(L.nt2, L.bn, smem_budget - epi_bytes, P.ov_nt2 ? P.ov_nt2 : kDefaultNT, L.kbps2 <= kDoubleAccMaxKb,
              L.ntu2, L.acc2);
    L.stage_bytes = gemm_stage_bytes(L.ntu1, L.bn);
    L.stages = std::min(kMaxStages, smem_budget / L.stage_bytes);
    if (P.ov_stages >= 2) L.stages = std::min(L.stages, P.ov_stages);
    L.smem = 3072 + L.stages * L.stage_bytes;
    L.stage_bytes2 = gemm_stage_bytes(L.ntu2, L.bn);
    L.stages2 = std::min(kMaxStages, (smem_budget - epi_bytes) / L.stage_bytes2);
    if (P.ov_stages >= 2) L.stages2 = std::min(L.stages2, P.ov_stages);
    L.smem2 = 3072 + epi_bytes + L.stages2 * L.stage_bytes2;
  }
  const int64_t units1 = static_cast<int64_t>(L.tiles_cap) * cdiv(L.nt1, L.ntu1) * L.s1;
  const int64_t units2 = static_cast<int64_t>(L.tiles_cap) * cdiv(L.nt2, L.ntu2) * L.s2;
  L.grid1 = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(P.num_sms, units1)));
  L.grid2 = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(P.num_sms, units2)));
  if (L.fused) L.grid1 = L.grid2 = P.num_sms * (L.fgroups == 1 ? 2 : 1);  // one queue for both GEMMs
  // split-K arrival counters; the fused launch adds its queue head (padded to
  // 32 entries), the ready counts of the route tiles and per-row-block counters
  // (and, always reserved so that the finalize switch never outgrows a
  // workspace, the finalize counters of T tokens x H / 16 column blocks)
  L.fix_len = 32 + L.tiles_cap + L.tiles_cap * L.nt1 * 8;
  L.ctr_len = L.fused ? L.fix_len + T * (d.hidden / 16) : L.tiles_cap * L.nt1;
  L.fin = L.fused && P.finalize;

  const int act_bytes = 2;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + std::max<size_t>(bytes, 1), 256);
    return at;
  };
  L.off_err = take(16);
  L.off_counts = take(sizeof(int32_t) * E);
  L.off_offs = take(sizeof(int32_t) * (E + 1));
  L.off_ntiles = take(sizeof(int32_t));
  L.off_tiles = take(sizeof(int32_t) * 4 * L.tiles_cap);
  L.off_perm = take(sizeof(int32_t) * L.slots_cap);
  L.off_inv = take(sizeof(int32_t) * std::max(L.R, 1));
  L.off_ctr = take(sizeof(int32_t) * L.ctr_len);
  L.off_chist = take(sizeof(int32_t) * kRouteMaxCtas * E);
  // gate/up split-K partials, or the tail pieces' (at most one per CTA)
  L.tail = (!L.gemv && L.s1 == 1 && P.tail_max > 1) ? P.tail_max : 0;
  L.off_part = take(L.s1 > 1 ? sizeof(float) * L.s1 * L.slots_cap * L.n1
                             : (L.tail ? sizeof(float) * L.grid1 * L.ntu1 * L.bn * 128 : 0));
  L.off_inter = take(static_cast<size_t>(act_bytes) * L.slots_cap * d.inter);
  // expert outputs: the activation dtype without down split-K, FP32 partials with it
  L.off_y = take((L.s2 == 1 ? static_cast<size_t>(act_bytes) : sizeof(float) * L.s2) * L.slots_cap * d.hidden);
  L.off_sx = take(static_cast<size_t>(act_bytes) * T * d.hidden);
  L.off_sids = take(sizeof(int32_t) * std::max(L.R, 1));
  L.off_sw = take(sizeof(float) * std::max(L.R, 1));
  L.off_sout = take(static_cast<size_t>(act_bytes) * T * d.hidden);
  L.total = o;
  return L;
}

size_t max_workspace(const w4a16_moe_plan_s& P) {
  size_t m = 0;
  for (int T = 1; T <= P.d.max_tokens; ++T) m = std::max(m, make_layout(P, T).total);
  return m;
}

// Route preparation CTAs: about 256 routes each (the per-CTA histogram pass
// is one route per thread), at most kRouteMaxCtas; with the router front end
// one token per warp.
void route_ctas(int T, int k, bool router, int& n_cta, int& tpc) {
  const int64_t want = router ? (T + kRoutePrepWarps - 1) / kRoutePrepWarps
                              : (static_cast<int64_t>(T) * k + 255) / 256;
  n_cta = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(kRouteMaxCtas, want)));
  tpc = std::max(1, (T + n_cta - 1) / n_cta);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Packed INT4 weights as a 3D uint8 tensor [E][rows][inner bytes], 128-byte
// swizzled boxes of 128 bytes x box_rows.
bool encode_weights(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t E,
                    uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, rows, E};
  cuuint64_t strides[2] = {inner, inner * rows};
  cuuint32_t box[3] = {128, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One whole 128-row weight tile per copy (the fused CUDA-core launch).
// Gated W13 with inter a multiple of 64: a 5D view [E][gate | up][I / 64][64
// rows][inner bytes], so that one box takes a tile's 64 gate rows and their 64
// up rows (inter rows apart) -- the view covers the tensor exactly.  Otherwise
// rows are contiguous: boxes of 128 rows of a 3D [E][rows][inner] view (rows
// past the end read as zero).  elem: 1 (packed bytes, 128-byte swizzle) or 2
// (BF16 scales, unswizzled); box_inner in elements.
bool encode_tile128(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t E, uint64_t gated_half,
                    int elem, uint32_t box_inner) {
  auto fn = encode_fn();
  if (!fn) return false;
  const CUtensorMapDataType t = elem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = elem == 1 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  const uint64_t row_bytes = inner * elem;
  if (gated_half != 0) {
    cuuint64_t dims[5] = {inner, 64, gated_half / 64, 2, E};
    cuuint64_t strides[4] = {row_bytes, 64 * row_bytes, gated_half * row_bytes, 2 * gated_half * row_bytes};
    cuuint32_t box[5] = {box_inner, 64, 1, 2, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, t, 5, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  cuuint64_t dims[3] = {inner, rows, E};
  cuuint64_t strides[2] = {row_bytes, row_bytes * rows};
  cuuint32_t box[3] = {box_inner, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, t, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Expert outputs y [rows][cols] (FP32, or the 16-bit activation dtype), unswizzled
// boxes of 32 columns x 16 rows (the down GEMM's output stores).
bool encode_out(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows, bool fp32, int dtype) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t es_bytes = fp32 ? 4 : 2;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * es_bytes};
  cuuint32_t box[2] = {32, 16};
  cuuint32_t es[2] = {1, 1};
  const CUtensorMapDataType t = fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : (dtype == W4A16_DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  return fn(m, t, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The masked-count layout's output [E][max_rows][H] as a 3D tensor with the
// same 32-column x 16-row boxes: a tile's rows past max_rows are dropped.
bool encode_out_masked(CUtensorMap* m, void* base, uint64_t cols, uint64_t max_rows, uint64_t E, int dtype) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cols, max_rows, E};
  cuuint64_t strides[2] = {cols * 2, cols * max_rows * 2};
  cuuint32_t box[3] = {32, 16, 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUtensorMapDataType t =
      dtype == W4A16_DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(m, t, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// BF16 group scales as a 3D tensor [E][rows][groups], unswizzled boxes of 8
// groups (16 bytes) x 64 rows; needs 16-byte aligned rows (groups % 8 == 0).
bool encode_scales(CUtensorMap* m, const void* base, uint64_t groups, uint64_t rows, uint64_t E) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {groups, rows, E};
  cuuint64_t strides[2] = {groups * 2, groups * rows * 2};
  cuuint32_t box[3] = {kGemvBlockK / kGroup, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A row-major 16-bit matrix [rows][cols], boxes of 64 columns x box_rows, 128B swizzle.
bool encode_rows16(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows,
                   int dtype) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dtype == W4A16_DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
            2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

w4a16_status validate_desc(const w4a16_moe_desc* d) {
  if (!d) return fail(W4A16_ERR_INVALID_ARG, "desc is NULL");
  if (d->num_experts < 1 || d->num_experts > 1024)
    return fail(W4A16_ERR_UNSUPPORTED, "num_experts must be in [1, 1024], got %d", d->num_experts);
  if (d->expert_offset < 0) return fail(W4A16_ERR_INVALID_ARG, "expert_offset must be >= 0");
  if (d->hidden <= 0 || d->hidden % 32 != 0)
    return fail(W4A16_ERR_UNSUPPORTED, "hidden must be a positive multiple of 32, got %d", d->hidden);
  if (d->inter <= 0 || d->inter % 32 != 0)
    return fail(W4A16_ERR_UNSUPPORTED, "inter must be a positive multiple of 32, got %d", d->inter);
  if (d->top_k < 1 || d->top_k > 16)
    return fail(W4A16_ERR_UNSUPPORTED, "top_k must be in [1, 16], got %d", d->top_k);
  if (d->max_tokens < 1 || d->max_tokens > 65536)
    return fail(W4A16_ERR_UNSUPPORTED, "max_tokens must be in [1, 65536], got %d", d->max_tokens);
  if (d->act != W4A16_ACT_SWIGLU && d->act != W4A16_ACT_RELU2)
    return fail(W4A16_ERR_INVALID_ARG, "unknown activation %d", d->act);
  if (d->scale_kind != W4A16_SCALE_GROUP32_K && d->scale_kind != W4A16_SCALE_PER_CHANNEL)
    return fail(W4A16_ERR_INVALID_ARG, "unknown scale kind %d", d->scale_kind);
  if (d->act_dtype != W4A16_DT_BF16 && d->act_dtype != W4A16_DT_FP16)
    return fail(W4A16_ERR_INVALID_ARG, "unknown activation dtype %d", d->act_dtype);
  if (d->global_experts != 0 && (d->global_experts < d->num_experts || d->global_experts > (1 << 20)))
    return fail(W4A16_ERR_INVALID_ARG, "global_experts must be 0 or in [num_experts, 2^20], got %d",
                d->global_experts);
  if (static_cast<int64_t>(d->max_tokens) * d->top_k > (1 << 24))
    return fail(W4A16_ERR_UNSUPPORTED, "max_tokens * top_k too large");
  return W4A16_OK;
}

w4a16_status check_ptr(const void* p, size_t align, const char* name) {
  if (!p) return fail(W4A16_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned(p, align)) return fail(W4A16_ERR_INVALID_ARG, "%s must be %zu-byte aligned", name, align);
  return W4A16_OK;
}

bool env_flag(const char* name, bool dflt) {
  const char* v = getenv(name);
  if (!v || !*v) return dflt;
  return !(v[0] == '0' && v[1] == 0);
}

// Route preparation for the ids of `ids`, or (logits != NULL) for the top-k
// of the router logits [T, G], whose ids / weights then go to ids_out /
// weights_out.
w4a16_status launch_prepare(const w4a16_moe_plan_s& P, const Layout& L, const int32_t* ids, uint8_t* ws,
                            cudaStream_t s, const float* logits = nullptr, int32_t G = 0,
                            int32_t* ids_out = nullptr, float* weights_out = nullptr) {
  RoutePrepParams rp = {};
  rp.ids = logits ? ids_out : ids;
  rp.T = L.T;
  rp.k = P.d.top_k;
  rp.E = P.d.num_experts;
  rp.expert_offset = P.d.expert_offset;
  rp.bm = L.bn;
  rp.counts = reinterpret_cast<int32_t*>(ws + L.off_counts);
  rp.offs = reinterpret_cast<int32_t*>(ws + L.off_offs);
  rp.perm = reinterpret_cast<int32_t*>(ws + L.off_perm);
  rp.inv = reinterpret_cast<int32_t*>(ws + L.off_inv);
  rp.tiles = reinterpret_cast<int4*>(ws + L.off_tiles);
  rp.num_tiles = reinterpret_cast<int32_t*>(ws + L.off_ntiles);
  rp.counters = reinterpret_cast<int32_t*>(ws + L.off_ctr);
  rp.ctr_len = L.ctr_len;
  rp.err = reinterpret_cast<int32_t*>(ws + L.off_err);
  rp.cta_hist = reinterpret_cast<int32_t*>(ws + L.off_chist);
  route_ctas(L.T, P.d.top_k, logits != nullptr, rp.n_cta, rp.tpc);
  rp.logits = logits;
  rp.G = G;
  rp.ids_out = ids_out;
  rp.weights_out = weights_out;
  cudaError_t e = launch_route_prep(rp, s, P.pdl);
  if (e != cudaSuccess) return cuda_fail(e, "route preparation launch");
  return W4A16_OK;
}

// Expert outputs -> output rows: the deterministic weighted combine.
w4a16_status launch_combine_of(const w4a16_moe_plan_s& P, const Layout& L, bool y16, const float* tw, int32_t renorm,
                               void* out, uint8_t* ws, cudaStream_t s) {
  CombineParams c = {};
  c.y = ws + L.off_y;
  c.y16 = y16 ? 1 : 0;
  c.slots_cap = L.slots_cap;
  c.splits = L.s2;
  c.inv = reinterpret_cast<const int32_t*>(ws + L.off_inv);
  c.topk_weights = tw;
  c.T = L.T;
  c.H = P.d.hidden;
  c.k = P.d.top_k;
  c.renormalize = renorm ? 1 : 0;
  c.out = out;
  if (L.fused) {
    c.zero = reinterpret_cast<int32_t*>(ws + L.off_ctr);
    c.zero_len = L.fix_len;
  }
  cudaError_t e = launch_combine(P.d.act_dtype, c, s, P.pdl);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  if (P.has_ev && (e = cudaEventRecord(P.ev[3], s)) != cudaSuccess) return cuda_fail(e, "event record");
  return W4A16_OK;
}

// CUDA-core path, both GEMMs in one launch (gemv_fused.cuh), then the combine.
// Gate rows per half of a gated W13 when the whole-tile 5D view applies
// (inter a multiple of 64), else 0.  The fused kernel takes the same decision.
uint64_t fused_gate_half(const w4a16_moe_desc& d) {
  return (d.act == W4A16_ACT_SWIGLU && d.inter % 64 == 0) ? static_cast<uint64_t>(d.inter) : 0;
}

w4a16_status launch_forward_fused(const w4a16_moe_plan_s& P, const Layout& L, const GemmParams& g,
                                  const GemmParams& g1, const CUtensorMap& tmA1, const CUtensorMap& tmS1,
                                  const CUtensorMap& tmA2, const CUtensorMap& tmS2, bool stma2, const uint8_t* w13,
                                  const uint16_t* s13, const uint8_t* w2, const uint16_t* s2, const float* tw,
                                  int32_t renorm, void* out, uint8_t* ws, cudaStream_t s) {
  const w4a16_moe_desc& d = P.d;
  FusedParams fp = {};
  fp.up = g1;
  fp.down = g;
  fp.down.n_rows = d.hidden;
  fp.down.K = d.inter;
  fp.down.out_cols = d.hidden;
  fp.down.n_tiles = L.nt2;
  fp.down.n_groups = L.nt2;
  fp.down.kb_total = L.kb2;
  fp.down.splits = 1;
  fp.down.kb_per_split = L.kb2;
  fp.down.x = ws + L.off_inter;
  fp.down.scales = s2;
  fp.down.out = ws + L.off_y;
  fp.down.scale_tma = stma2 ? 1 : 0;
  fp.down.out16 = 1;
  int32_t* ctr = reinterpret_cast<int32_t*>(ws + L.off_ctr);
  fp.queue = ctr;
  fp.ready = ctr + 32;
  fp.fix = ctr + 32 + L.tiles_cap;
  fp.down_chunk = L.down_chunk;
  fp.groups = L.fgroups;
  if (L.fin) {
    fp.finalize = 1;
    fp.fin_ctr = ctr + L.fix_len;
    fp.inv = reinterpret_cast<const int32_t*>(ws + L.off_inv);
    fp.topk_weights = tw;
    fp.T = L.T;
    fp.k = d.top_k;
    fp.renormalize = renorm ? 1 : 0;
    fp.out = out;
    fp.exit_ctr = ctr + 1;  // inside the queue head's padding, so reset with it
    fp.reset = ctr;
    fp.reset_len = L.fix_len;
  }
  const int lay = P.layout == W4A16_LAYOUT_INTERLEAVED ? LAYOUT_IL : LAYOUT_CANON;
  // whole-tile copies (one box per weight tile and stage) for the K-packed
  // layouts; the per-channel row-pair layout keeps its four boxes
  CUtensorMap wA1 = tmA1, wS1 = tmS1, wA2 = tmA2, wS2 = tmS2;
  const bool group = d.scale_kind == W4A16_SCALE_GROUP32_K;
  if (group || lay == LAYOUT_IL) {
    const uint64_t half = fused_gate_half(d);
    // gated W13 whose inter is an odd multiple of 32 keeps its 64-row boxes
    // (a tile's halves are neither consecutive nor a whole 5D view)
    const bool up_whole = d.act != W4A16_ACT_SWIGLU || half != 0;
    bool ok = !up_whole || encode_tile128(&wA1, w13, d.hidden / 2, L.n1, d.num_experts, half, 1, 128);
    ok = ok && encode_tile128(&wA2, w2, d.inter / 2, d.hidden, d.num_experts, 0, 1, 128);
    if (ok && up_whole && fp.up.scale_tma)
      ok = encode_tile128(&wS1, s13, d.hidden / kGroup, L.n1, d.num_experts, half, 2, 8);
    if (ok && fp.down.scale_tma) ok = encode_tile128(&wS2, s2, d.inter / kGroup, d.hidden, d.num_experts, 0, 2, 8);
    if (!ok) return fail(W4A16_ERR_CUDA, "cuTensorMapEncodeTiled failed (whole-tile weight boxes)");
  }
  cudaError_t e =
      launch_gemv_fused(d.scale_kind, d.act_dtype, lay, fp, wA1, wS1, wA2, wS2, L.grid1, L.smem, s, P.pdl);
  if (e != cudaSuccess) return cuda_fail(e, "fused expert GEMM launch");
  // both GEMMs end with the one launch: the gate/up and down stage marks coincide
  if (P.has_ev && ((e = cudaEventRecord(P.ev[1], s)) != cudaSuccess || (e = cudaEventRecord(P.ev[2], s)) != cudaSuccess))
    return cuda_fail(e, "event record");
  if (L.fin) {
    if (P.has_ev && (e = cudaEventRecord(P.ev[3], s)) != cudaSuccess) return cuda_fail(e, "event record");
    return W4A16_OK;
  }
  return launch_combine_of(P, L, true, tw, renorm, out, ws, s);
}

// masked_rows > 0: the masked-count layout's [E][masked_rows][H] output, which
// the tensor-core down GEMM (without split-K) writes directly -- its single
// unit-weight route per row needs no combine; rows past the counts are then
// zeroed.  Other paths combine as usual.
w4a16_status launch_forward(const w4a16_moe_plan_s& P, const Layout& L, const void* x,
                            const uint8_t* w13, const uint16_t* s13, const uint8_t* w2,
                            const uint16_t* s2, const float* tw, int32_t renorm, void* out,
                            uint8_t* ws, cudaStream_t s, int32_t masked_rows = 0) {
  const w4a16_moe_desc& d = P.d;
  const bool group = d.scale_kind == W4A16_SCALE_GROUP32_K;
  const bool il = P.layout == W4A16_LAYOUT_INTERLEAVED;
  CUtensorMap tmA1, tmA2, tmB2;
  bool ok;
  if (group || il) {
    // rows of packed bytes along K; boxes of 64 rows x one stage of K (128
    // bytes = 256 K values, 128-byte swizzle) on both paths
    static_assert(kGemvBlockK / 2 == 128 && kBlockK / 2 == 128, "weight boxes are 128 bytes wide");
    ok = encode_weights(&tmA1, w13, d.hidden / 2, L.n1, d.num_experts, 64) &&
         encode_weights(&tmA2, w2, d.inter / 2, d.hidden, d.num_experts, 64);
  } else {
    // row pairs of K bytes; boxes of 128 bytes (128 K values) x 32 row pairs
    ok = encode_weights(&tmA1, w13, d.hidden, L.n1 / 2, d.num_experts, 32) &&
         encode_weights(&tmA2, w2, d.inter, d.hidden / 2, d.num_experts, 32);
  }
  ok = ok && encode_rows16(&tmB2, ws + L.off_inter, d.inter, L.slots_cap, L.bn, d.act_dtype);
  // the tensor-core gate/up GEMM gathers its activation rows itself (no map)
  CUtensorMap tmNone;
  memset(&tmNone, 0, sizeof(tmNone));
  // tensor-core path: expert outputs y [splits * slots_cap, H], TMA-stored
  const bool y16 = L.s2 == 1;
  const bool masked_direct = masked_rows > 0 && !L.gemv && y16;
  CUtensorMap tmY;
  memset(&tmY, 0, sizeof(tmY));
  if (masked_direct)
    ok = ok && encode_out_masked(&tmY, out, d.hidden, masked_rows, d.num_experts, d.act_dtype);
  else if (!L.gemv)
    ok = ok && encode_out(&tmY, ws + L.off_y, d.hidden, static_cast<uint64_t>(L.s2) * L.slots_cap, !y16, d.act_dtype);
  // group scales by TMA (boxes of 8 groups) where their rows are 16-byte multiples
  CUtensorMap tmS1, tmS2;
  memset(&tmS1, 0, sizeof(tmS1));
  memset(&tmS2, 0, sizeof(tmS2));
  const bool stma1 = group && (d.hidden / kGroup) % 8 == 0 && aligned(s13, 16);
  const bool stma2 = group && (d.inter / kGroup) % 8 == 0 && aligned(s2, 16);
  if (stma1) ok = ok && encode_scales(&tmS1, s13, d.hidden / kGroup, L.n1, d.num_experts);
  if (stma2) ok = ok && encode_scales(&tmS2, s2, d.inter / kGroup, d.hidden, d.num_experts);
  if (!ok) return fail(W4A16_ERR_CUDA, "cuTensorMapEncodeTiled failed (driver entry point or arguments)");
  // tensor-core path: whole-tile boxes for the K-packed layouts (one copy per
  // 128-row weight tile and stage; see encode_tile128)
  if (!L.gemv && (group || il)) {
    const uint64_t half = fused_gate_half(d);
    const bool up_whole = d.act != W4A16_ACT_SWIGLU || half != 0;
    ok = (!up_whole || encode_tile128(&tmA1, w13, d.hidden / 2, L.n1, d.num_experts, half, 1, 128)) &&
         encode_tile128(&tmA2, w2, d.inter / 2, d.hidden, d.num_experts, 0, 1, 128);
    if (ok && up_whole && stma1) ok = encode_tile128(&tmS1, s13, d.hidden / kGroup, L.n1, d.num_experts, half, 2, 8);
    if (ok && stma2) ok = encode_tile128(&tmS2, s2, d.inter / kGroup, d.hidden, d.num_experts, 0, 2, 8);
    if (!ok) return fail(W4A16_ERR_CUDA, "cuTensorMapEncodeTiled failed (whole-tile weight boxes)");
  }

  GemmParams g = {};
  g.act = d.act;
  g.E = d.num_experts;
  g.inter = d.inter;
  g.bn = L.bn;
  g.stages = L.stages;
  g.stage_bytes = L.stage_bytes;
  g.top_k = d.top_k;
  g.tiles = reinterpret_cast<const int4*>(ws + L.off_tiles);
  g.num_tiles = reinterpret_cast<const int32_t*>(ws + L.off_ntiles);
  g.perm = reinterpret_cast<const int32_t*>(ws + L.off_perm);
  g.slots_cap = L.slots_cap;
  g.err = reinterpret_cast<int32_t*>(ws + L.off_err);
  g.tiles_cap = L.tiles_cap;
  g.wait_ns = P.wait_ns;
  const int lay = il ? LAYOUT_IL : LAYOUT_CANON;

  GemmParams g1 = g;
  g1.nt_unit = L.ntu1;
  g1.n_groups = cdiv(L.nt1, L.ntu1);
  g1.acc_bufs = L.acc1;
  g1.n_rows = L.n1;
  g1.K = d.hidden;
  g1.out_cols = d.inter;
  g1.n_tiles = L.nt1;
  g1.kb_total = L.kb1;
  g1.splits = L.s1;
  g1.kb_per_split = L.kbps1;
  g1.x = x;
  g1.scales = s13;
  g1.out = ws + L.off_inter;
  g1.part = reinterpret_cast<float*>(ws + L.off_part);
  g1.counters = reinterpret_cast<int32_t*>(ws + L.off_ctr);
  g1.tail_max = L.tail;
  g1.scale_tma = stma1 ? 1 : 0;
  cudaError_t e;
  if (P.has_ev && (e = cudaEventRecord(P.ev[0], s)) != cudaSuccess) return cuda_fail(e, "event record");
  if (L.fused)
    return launch_forward_fused(P, L, g, g1, tmA1, tmS1, tmA2, tmS2, stma2, w13, s13, w2, s2, tw, renorm, out, ws, s);
  e = L.gemv ? launch_gemv(GEMM_UP, d.scale_kind, d.act_dtype, lay, g1, tmA1, tmS1, L.grid1, L.smem, s, P.pdl)
             : launch_gemm(GEMM_UP, d.scale_kind, d.act_dtype, lay, g1, tmA1, tmNone, tmY, tmS1, L.grid1, L.smem, s,
                           P.pdl);
  if (e != cudaSuccess) return cuda_fail(e, "gate/up GEMM launch");
  if (P.has_ev && (e = cudaEventRecord(P.ev[1], s)) != cudaSuccess) return cuda_fail(e, "event record");

  GemmParams g2 = g;
  g2.stages = L.stages2;
  if (!L.gemv) g2.stage_bytes = L.stage_bytes2;
  g2.nt_unit = L.ntu2;
  g2.n_groups = cdiv(L.nt2, L.ntu2);
  g2.acc_bufs = L.acc2;
  g2.n_rows = d.hidden;
  g2.K = d.inter;
  g2.out_cols = d.hidden;
  g2.n_tiles = L.nt2;
  g2.kb_total = L.kb2;
  g2.splits = L.s2;
  g2.kb_per_split = L.kbps2;
  g2.x = ws + L.off_inter;
  g2.scales = s2;
  g2.out = ws + L.off_y;
  g2.part = nullptr;
  g2.counters = nullptr;
  g2.scale_tma = stma2 ? 1 : 0;
  g2.out16 = y16 ? 1 : 0;
  g2.masked_rows = masked_direct ? masked_rows : 0;
  g2.seg_offs = masked_direct ? reinterpret_cast<const int32_t*>(ws + L.off_offs) : nullptr;
  e = L.gemv ? launch_gemv(GEMM_DOWN, d.scale_kind, d.act_dtype, lay, g2, tmA2, tmS2, L.grid2, L.smem2, s, P.pdl)
             : launch_gemm(GEMM_DOWN, d.scale_kind, d.act_dtype, lay, g2, tmA2, tmB2, tmY, tmS2, L.grid2, L.smem2, s,
                           P.pdl);
  if (e != cudaSuccess) return cuda_fail(e, "down GEMM launch");
  if (P.has_ev && (e = cudaEventRecord(P.ev[2], s)) != cudaSuccess) return cuda_fail(e, "event record");

  if (masked_direct) {
    e = launch_masked_zero_rows(reinterpret_cast<const int32_t*>(ws + L.off_counts), d.num_experts, masked_rows,
                                d.hidden, out, s, P.pdl);
    if (e != cudaSuccess) return cuda_fail(e, "masked zero-rows launch");
    if (P.has_ev && (e = cudaEventRecord(P.ev[3], s)) != cudaSuccess) return cuda_fail(e, "event record");
    return W4A16_OK;
  }
  return launch_combine_of(P, L, y16, tw, renorm, out, ws, s);
}

}  // namespace

namespace w4a16 {
template <int DT, int LAYOUT>
cudaError_t launch_gemm_dt(int which, int scale_kind, const GemmParams& p, const CUtensorMap& tmA,
                           const CUtensorMap& tmB, const CUtensorMap& tmC, const CUtensorMap& tmS,
                           int grid, int smem_bytes, cudaStream_t s, bool pdl);
#define W4A16_GEMM_EXTERN(DT, LAYOUT)                                                                          \
  extern template cudaError_t launch_gemm_dt<DT, LAYOUT>(int, int, const GemmParams&, const CUtensorMap&,     \
                                                         const CUtensorMap&, const CUtensorMap&,              \
                                                         const CUtensorMap&, int, int, cudaStream_t, bool);
W4A16_GEMM_EXTERN(DT_BF16, LAYOUT_CANON)
W4A16_GEMM_EXTERN(DT_FP16, LAYOUT_CANON)
W4A16_GEMM_EXTERN(DT_BF16, LAYOUT_IL)
W4A16_GEMM_EXTERN(DT_FP16, LAYOUT_IL)
#undef W4A16_GEMM_EXTERN

cudaError_t launch_gemm(int which, int scale_kind, int dtype, int layout, const GemmParams& p,
                        const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                        const CUtensorMap& tmS, int grid, int smem_bytes, cudaStream_t s, bool pdl) {
  if (layout == LAYOUT_IL)
    return dtype == DT_BF16
               ? launch_gemm_dt<DT_BF16, LAYOUT_IL>(which, scale_kind, p, tmA, tmB, tmC, tmS, grid, smem_bytes, s, pdl)
               : launch_gemm_dt<DT_FP16, LAYOUT_IL>(which, scale_kind, p, tmA, tmB, tmC, tmS, grid, smem_bytes, s, pdl);
  return dtype == DT_BF16
             ? launch_gemm_dt<DT_BF16, LAYOUT_CANON>(which, scale_kind, p, tmA, tmB, tmC, tmS, grid, smem_bytes, s, pdl)
             : launch_gemm_dt<DT_FP16, LAYOUT_CANON>(which, scale_kind, p, tmA, tmB, tmC, tmS, grid, smem_bytes, s, pdl);
}

template <int DT, int LAYOUT>
cudaError_t launch_gemv_dt(int which, int scale_kind, const GemmParams& p, const CUtensorMap& tmA,
                           const CUtensorMap& tmS, int grid, int smem_bytes, cudaStream_t s, bool pdl);
#define W4A16_GEMV_EXTERN(DT, LAYOUT)                                                                          \
  extern template cudaError_t launch_gemv_dt<DT, LAYOUT>(int, int, const GemmParams&, const CUtensorMap&,     \
                                                         const CUtensorMap&, int, int, cudaStream_t, bool);
W4A16_GEMV_EXTERN(DT_BF16, LAYOUT_CANON)
W4A16_GEMV_EXTERN(DT_FP16, LAYOUT_CANON)
W4A16_GEMV_EXTERN(DT_BF16, LAYOUT_IL)
W4A16_GEMV_EXTERN(DT_FP16, LAYOUT_IL)
#undef W4A16_GEMV_EXTERN

cudaError_t launch_gemv(int which, int scale_kind, int dtype, int layout, const GemmParams& p, const CUtensorMap& tmA,
                        const CUtensorMap& tmS, int grid, int smem_bytes, cudaStream_t s, bool pdl) {
  if (layout == LAYOUT_IL)
    return dtype == DT_BF16 ? launch_gemv_dt<DT_BF16, LAYOUT_IL>(which, scale_kind, p, tmA, tmS, grid, smem_bytes, s, pdl)
                            : launch_gemv_dt<DT_FP16, LAYOUT_IL>(which, scale_kind, p, tmA, tmS, grid, smem_bytes, s, pdl);
  return dtype == DT_BF16 ? launch_gemv_dt<DT_BF16, LAYOUT_CANON>(which, scale_kind, p, tmA, tmS, grid, smem_bytes, s, pdl)
                          : launch_gemv_dt<DT_FP16, LAYOUT_CANON>(which, scale_kind, p, tmA, tmS, grid, smem_bytes, s, pdl);
}

template <int DT, int LAYOUT>
cudaError_t launch_gemv_fused_dt(int scale_kind, const FusedParams& fp, const CUtensorMap& tmA1,
                                 const CUtensorMap& tmS1, const CUtensorMap& tmA2, const CUtensorMap& tmS2, int grid,
                                 int smem_bytes, cudaStream_t s, bool pdl);
#define W4A16_FUSED_EXTERN(DT, LAYOUT)                                                                          \
  extern template cudaError_t launch_gemv_fused_dt<DT, LAYOUT>(int, const FusedParams&, const CUtensorMap&,    \
                                                               const CUtensorMap&, const CUtensorMap&,         \
                                                               const CUtensorMap&, int, int, cudaStream_t, bool);
W4A16_FUSED_EXTERN(DT_BF16, LAYOUT_CANON)
W4A16_FUSED_EXTERN(DT_FP16, LAYOUT_CANON)
W4A16_FUSED_EXTERN(DT_BF16, LAYOUT_IL)
W4A16_FUSED_EXTERN(DT_FP16, LAYOUT_IL)
#undef W4A16_FUSED_EXTERN

cudaError_t launch_gemv_fused(int scale_kind, int dtype, int layout, const FusedParams& p, const CUtensorMap& tmA1,
                              const CUtensorMap& tmS1, const CUtensorMap& tmA2, const CUtensorMap& tmS2, int grid,
                              int smem_bytes, cudaStream_t s, bool pdl) {
  if (layout == LAYOUT_IL)
    return dtype == DT_BF16
               ? launch_gemv_fused_dt<DT_BF16, LAYOUT_IL>(scale_kind, p, tmA1, tmS1, tmA2, tmS2, grid, smem_bytes, s, pdl)
               : launch_gemv_fused_dt<DT_FP16, LAYOUT_IL>(scale_kind, p, tmA1, tmS1, tmA2, tmS2, grid, smem_bytes, s, pdl);
  return dtype == DT_BF16
             ? launch_gemv_fused_dt<DT_BF16, LAYOUT_CANON>(scale_kind, p, tmA1, tmS1, tmA2, tmS2, grid, smem_bytes, s, pdl)
             : launch_gemv_fused_dt<DT_FP16, LAYOUT_CANON>(scale_kind, p, tmA1, tmS1, tmA2, tmS2, grid, smem_bytes, s, pdl);
}
}  // namespace w4a16

extern "C" {

w4a16_status w4a16_moe_plan(const w4a16_moe_desc* desc, w4a16_moe_plan_t* out, size_t* workspace_bytes) {
  if (!out || !workspace_bytes) return fail(W4A16_ERR_INVALID_ARG, "out / workspace_bytes is NULL");
  *out = nullptr;
  w4a16_status st = validate_desc(desc);
  if (st != W4A16_OK) return st;
  auto* P = new w4a16_moe_plan_s();
  P->d = *desc;
  P->num_sms = 152;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0) {
    P->num_sms = sms;
  } else {
    cudaGetLastError();  // no device here: plan with the GB300 SM count
  }
  P->pdl = env_flag("W4A16_MOE_PDL", true);
  P->fused = env_flag("W4A16_MOE_FUSED", true);
  P->finalize = env_flag("W4A16_MOE_FUSED_FINALIZE", false);
  if (const char* v = getenv("W4A16_MOE_DOWN_CHUNK")) P->ov_chunk = std::max(0, atoi(v));
  P->tail_max = kDefaultTailPieces;
  if (const char* v = getenv("W4A16_MOE_TAIL_PIECES")) P->tail_max = std::min(std::max(0, atoi(v)), 64);
  P->layout = W4A16_LAYOUT_CHECKPOINT;
  // tuning knobs for measurements: weight tiles per tensor-core unit of each GEMM
  if (const char* v = getenv("W4A16_MOE_NT_GATE_UP")) P->ov_nt1 = atoi(v);
  if (const char* v = getenv("W4A16_MOE_NT_DOWN")) P->ov_nt2 = atoi(v);
  if (const char* v = getenv("W4A16_MOE_TC_STAGES")) P->ov_stages = atoi(v);
  if (const char* v = getenv("W4A16_MOE_CC_TILE_ROWS")) P->ov_bn_cc = atoi(v);
  if (const char* v = getenv("W4A16_MOE_FUSED_GROUPS")) P->ov_fgroups = atoi(v);
  if (P->ov_nt1 != 0 && P->ov_nt1 != 1 && P->ov_nt1 != 2 && P->ov_nt1 != 4) P->ov_nt1 = 0;
  if (P->ov_nt2 != 0 && P->ov_nt2 != 1 && P->ov_nt2 != 2 && P->ov_nt2 != 4) P->ov_nt2 = 0;
  P->wait_ns = kWaitTimeoutNs;
  if (const char* v = getenv("W4A16_MOE_WAIT_TIMEOUT_NS")) {
    const unsigned long long ns = strtoull(v, nullptr, 10);
    if (ns > 0) P->wait_ns = ns;
  }
  P->ws_bytes = max_workspace(*P);
  *out = P;
  *workspace_bytes = P->ws_bytes;
  return W4A16_OK;
}

w4a16_status w4a16_moe_plan_destroy(w4a16_moe_plan_t plan) {
  delete plan;
  return W4A16_OK;
}

w4a16_status w4a16_moe_set_overrides(w4a16_moe_plan_t plan, int32_t tile_rows, int32_t s1, int32_t s2,
                                     size_t* workspace_bytes) {
  if (!plan) return fail(W4A16_ERR_INVALID_ARG, "plan is NULL");
  if (tile_rows != 0 && (tile_rows < 16 || tile_rows > kMaxBN || tile_rows % 16 != 0))
    return fail(W4A16_ERR_INVALID_ARG, "tile_rows must be 0 or a multiple of 16 in [16, %d]", kMaxBN);
  if (s1 < 0 || s1 > 64 || s2 < 0 || s2 > 64)
    return fail(W4A16_ERR_INVALID_ARG, "split factors must be in [0, 64]");
  plan->ov_bn = tile_rows;
  plan->ov_s1 = s1;
  plan->ov_s2 = s2;
  plan->ws_bytes = max_workspace(*plan);
  if (workspace_bytes) *workspace_bytes = plan->ws_bytes;
  return W4A16_OK;
}

w4a16_status w4a16_moe_set_gemm_path(w4a16_moe_plan_t plan, int32_t path, size_t* workspace_bytes) {
  if (!plan) return fail(W4A16_ERR_INVALID_ARG, "plan is NULL");
  if (path != W4A16_PATH_AUTO && path != W4A16_PATH_TENSOR_CORES && path != W4A16_PATH_CUDA_CORES)
    return fail(W4A16_ERR_INVALID_ARG, "unknown GEMM path %d", path);
  plan->path = path;
  plan->ws_bytes = max_workspace(*plan);
  if (workspace_bytes) *workspace_bytes = plan->ws_bytes;
  return W4A16_OK;
}

w4a16_status w4a16_moe_route_info(w4a16_moe_plan_t plan, int32_t num_tokens, w4a16_route_info* info) {
  if (!plan || !info) return fail(W4A16_ERR_INVALID_ARG, "plan / info is NULL");
  if (num_tokens < 0 || num_tokens > plan->d.max_tokens)
    return fail(W4A16_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", num_tokens, plan->d.max_tokens);
  const Layout L = make_layout(*plan, num_tokens);
  info->tile_rows = L.bn;
  info->max_slots = static_cast<int32_t>(L.slots_cap);
  info->max_tiles = L.tiles_cap;
  info->gemm1_splits = L.s1;
  info->gemm2_splits = L.s2;
  info->gemm1_ctas = L.grid1;
  info->gemm2_ctas = L.grid2;
  info->pipeline_stages = L.stages;
  info->gemm_path = L.gemv ? W4A16_PATH_CUDA_CORES : W4A16_PATH_TENSOR_CORES;
  info->fused_gemms = L.fused ? 1 : 0;
  info->fused_finalize = L.fin ? 1 : 0;
  info->off_counts = L.off_counts;
  info->off_offs = L.off_offs;
  info->off_perm = L.off_perm;
  info->off_inv = L.off_inv;
  info->off_tiles = L.off_tiles;
  info->off_num_tiles = L.off_ntiles;
  info->off_inter = L.off_inter;
  info->off_expert_out = L.off_y;
  return W4A16_OK;
}

w4a16_status w4a16_moe_prepare_routes(w4a16_moe_plan_t plan, int32_t num_tokens, const int32_t* topk_ids,
                                      void* workspace, void* stream) {
  if (!plan) return fail(W4A16_ERR_INVALID_ARG, "plan is NULL");
  if (num_tokens < 0 || num_tokens > plan->d.max_tokens)
    return fail(W4A16_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", num_tokens, plan->d.max_tokens);
  if (num_tokens == 0) return W4A16_OK;
  w4a16_status st;
  if ((st = check_ptr(topk_ids, 4, "topk_ids")) != W4A16_OK) return st;
  if ((st = check_ptr(workspace, 256, "workspace")) != W4A16_OK) return st;
  const Layout L = make_layout(*plan, num_tokens);
  return launch_prepare(*plan, L, topk_ids, static_cast<uint8_t*>(workspace),
                        static_cast<cudaStream_t>(stream));
}

w4a16_status w4a16_moe_forward(w4a16_moe_plan_t plan, int32_t num_tokens, const void* x, const uint8_t* w13,
                               const uint16_t* s13, const uint8_t* w2, const uint16_t* s2,
                               const float* topk_weights, const int32_t* topk_ids, int32_t renormalize,
                               void* out, void* workspace, void* stream) {
  if (!plan) return fail(W4A16_ERR_INVALID_ARG, "plan is NULL");
  if (num_tokens < 0 || num_tokens > plan->d.max_tokens)
    return fail(W4A16_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", num_tokens, plan->d.max_tokens);
  if (num_tokens == 0) return W4A16_OK;
  w4a16_status st;
  if ((st = check_ptr(x, 16, "x")) != W4A16_OK) return st;
  if ((st = check_ptr(w13, 16, "w13")) != W4A16_OK) return st;
  if ((st = check_ptr(s13, 4, "s13")) != W4A16_OK) return st;
  if ((st = check_ptr(w2, 16, "w2")) != W4A16_OK) return st;
  if ((st = check_ptr(s2, 4, "s2")) != W4A16_OK) return st;
  if ((st = check_ptr(topk_weights, 4, "topk_weights")) != W4A16_OK) return st;
  if ((st = check_ptr(topk_ids, 4, "topk_ids")) != W4A16_OK) return st;
  if ((st = check_ptr(out, 16, "out")) != W4A16_OK) return st;
  if ((st = check_ptr(workspace, 256, "workspace")) != W4A16_OK) return st;
  const Layout L = make_layout(*plan, num_tokens);
  return launch_forward(*plan, L, x, w13, s13, w2, s2, topk_weights, renormalize, out,
                        static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream));
}

w4a16_status w4a16_moe_forward_host(w4a16_moe_plan_t plan, int32_t num_tokens, const void* x_host,
                                    const uint8_t* w13, const uint16_t* s13, const uint8_t* w2,
                                    const uint16_t* s2, const float* topk_weights_host,
                                    const int32_t* topk_ids_host, int32_t renormalize, void* out_host,
                                    void* workspace, void* stream) {
  if (!plan) return fail(W4A16_ERR_INVALID_ARG, "plan is NULL");
  if (num_tokens < 0 || num_tokens > plan->d.max_tokens)
    return fail(W4A16_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", num_tokens, plan->d.max_tokens);
  if (num_tokens == 0) return W4A16_OK;
  if (!x_host || !topk_weights_host || !topk_ids_host || !out_host)
    return fail(W4A16_ERR_INVALID_ARG, "host buffer is NULL");
  w4a16_status st;
  if ((st = check_ptr(workspace, 256, "workspace")) != W4A16_OK) return st;
  const Layout L = make_layout(*plan, num_tokens);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t xb = static_cast<size_t>(num_tokens) * plan->d.hidden * 2;
  const size_t rb = static_cast<size_t>(L.R) * 4;
  cudaError_t e;
  if ((e = cudaMemcpyAsync(ws + L.off_sx, x_host, xb, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "copy x");
  if ((e = cudaMemcpyAsync(ws + L.off_sids, topk_ids_host, rb, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "copy topk_ids");
  if ((e = cudaMemcpyAsync(ws + L.off_sw, topk_weights_host, rb, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "copy topk_weights");
  st = w4a16_moe_prepare_routes(plan, num_tokens, reinterpret_cast<const int32_t*>(ws + L.off_sids), workspace,
                                stream);
  if (st != W4A16_OK) return st;
  st = w4a16_moe_forward(plan, num_tokens, ws + L.off_sx, w13, s13, w2, s2,
                         reinterpret_cast<const float*>(ws + L.off_sw),
                         reinterpret_cast<const int32_t*>(ws + L.off_sids), renormalize, ws + L.off_sout,
                         workspace, stream);
  if (st != W4A16_OK) return st;
  if ((e = cudaMemcpyAsync(out_host, ws + L.off_sout, xb, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(e, "copy out");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "stream sync");
  return W4A16_OK;
}

namespace {
w4a16_status static_workspace_ptr(void** out);
}

w4a16_status w4a16_moe_check_device_error(w4a16_moe_plan_t plan, void* workspace, void* stream) {
  if (!plan) return fail(W4A16_ERR_INVALID_ARG, "plan is NULL");
  if (!workspace) {
    // the fixed workspace of w4a16_moe_forward_static_workspace
    w4a16_status st = static_workspace_ptr(&workspace);
    if (st != W4A16_OK) return st;
  }
  const Layout L = make_layout(*plan, 1);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t flag = 0;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaMemcpyAsync(&flag, ws + L.off_err, sizeof(flag), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "read device error flag");
  if (flag != 0) {
    e = cudaMemsetAsync(ws + L.off_err, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return fail(W4A16_ERR_DEVICE_TIMEOUT, "a bounded wait inside a kernel timed out (flag %d)", flag);
  }
  return W4A16_OK;
}

w4a16_status w4a16_moe_forward_masked(w4a16_moe_plan_t plan, int32_t max_rows, const int32_t* counts,
                                      const void* x, const uint8_t* w13, const uint16_t* s13, const uint8_t* w2,
                                      const uint16_t* s2, void* y, void* workspace, void* stream) {
  if (!plan) return fail(W4A16_ERR_INVALID_ARG, "plan is NULL");
  if (plan->d.top_k != 1)
    return fail(W4A16_ERR_UNSUPPORTED, "the masked-count layout routes every row once: the plan needs top_k == 1, got %d",
                plan->d.top_k);
  if (max_rows < 0) return fail(W4A16_ERR_INVALID_ARG, "max_rows must be >= 0, got %d", max_rows);
  const int64_t rows = static_cast<int64_t>(plan->d.num_experts) * max_rows;
  if (rows > plan->d.max_tokens)
    return fail(W4A16_ERR_INVALID_ARG, "num_experts * max_rows = %lld exceeds the plan's max_tokens %d",
                static_cast<long long>(rows), plan->d.max_tokens);
  if (rows == 0) return W4A16_OK;
  w4a16_status st;
  if ((st = check_ptr(counts, 4, "counts")) != W4A16_OK) return st;
  if ((st = check_ptr(workspace, 256, "workspace")) != W4A16_OK) return st;
  const int32_t T = static_cast<int32_t>(rows);
  const Layout L = make_layout(*plan, T);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* ids = reinterpret_cast<int32_t*>(ws + L.off_sids);
  float* wts = reinterpret_cast<float*>(ws + L.off_sw);
  cudaError_t e = launch_masked_routes(counts, plan->d.num_experts, max_rows, plan->d.expert_offset, ids, wts,
                                       plan->num_sms, static_cast<cudaStream_t>(stream), plan->pdl);
  if (e != cudaSuccess) return cuda_fail(e, "masked-route launch");
  st = w4a16_moe_prepare_routes(plan, T, ids, workspace, stream);
  if (st != W4A16_OK) return st;
  if ((st = check_ptr(x, 16, "x")) != W4A16_OK) return st;
  if ((st = check_ptr(w13, 16, "w13")) != W4A16_OK) return st;
  if ((st = check_ptr(s13, 4, "s13")) != W4A16_OK) return st;
  if ((st = check_ptr(w2, 16, "w2")) != W4A16_OK) return st;
  if ((st = check_ptr(s2, 4, "s2")) != W4A16_OK) return st;
  if ((st = check_ptr(y, 16, "y")) != W4A16_OK) return st;
  // the rows' single unit-weight routes: the tensor-core down GEMM writes y
  // directly (no combine), other paths combine into it
  return launch_forward(*plan, L, x, w13, s13, w2, s2, wts, 0, y, ws, static_cast<cudaStream_t>(stream), max_rows);
}

w4a16_status w4a16_moe_route_topk(const float* logits, int32_t num_tokens, int32_t num_global, int32_t top_k,
                                  int32_t* topk_ids, float* topk_weights, void* stream) {
  if (num_tokens < 0) return fail(W4A16_ERR_INVALID_ARG, "num_tokens must be >= 0, got %d", num_tokens);
  if (num_global < 1 || num_global > 1024)
    return fail(W4A16_ERR_UNSUPPORTED, "num_global must be in [1, 1024], got %d", num_global);
  if (top_k < 1 || top_k > 16 || top_k > num_global)
    return fail(W4A16_ERR_UNSUPPORTED, "top_k must be in [1, min(16, num_global)], got %d", top_k);
  if (num_tokens == 0) return W4A16_OK;
  w4a16_status st;
  if ((st = check_ptr(logits, 4, "logits")) != W4A16_OK) return st;
  if ((st = check_ptr(topk_ids, 4, "topk_ids")) != W4A16_OK) return st;
  if ((st = check_ptr(topk_weights, 4, "topk_weights")) != W4A16_OK) return st;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  w4a16::RouterParams rp;
  rp.logits = logits;
  rp.T = num_tokens;
  rp.G = num_global;
  rp.k = top_k;
  rp.ids = topk_ids;
  rp.weights = topk_weights;
  e = w4a16::launch_router(rp, sms, static_cast<cudaStream_t>(stream), env_flag("W4A16_MOE_PDL", true));
  if (e != cudaSuccess) return cuda_fail(e, "router launch");
  return W4A16_OK;
}

w4a16_status w4a16_moe_route_and_prepare(w4a16_moe_plan_t plan, int32_t num_tokens, const float* logits,
                                         int32_t num_global, int32_t* topk_ids, float* topk_weights, void* workspace,
                                         void* stream) {
  if (!plan) return fail(W4A16_ERR_INVALID_ARG, "plan is NULL");
  if (num_tokens < 0 || num_tokens > plan->d.max_tokens)
    return fail(W4A16_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", num_tokens, plan->d.max_tokens);
  if (num_global < 1 || num_global > 1024)
    return fail(W4A16_ERR_UNSUPPORTED, "num_global must be in [1, 1024], got %d", num_global);
  if (plan->d.top_k > num_global)
    return fail(W4A16_ERR_UNSUPPORTED, "top_k %d exceeds num_global %d", plan->d.top_k, num_global);
  if (num_tokens == 0) return W4A16_OK;
  w4a16_status st;
  if ((st = check_ptr(logits, 4, "logits")) != W4A16_OK) return st;
  if ((st = check_ptr(topk_ids, 4, "topk_ids")) != W4A16_OK) return st;
  if ((st = check_ptr(topk_weights, 4, "topk_weights")) != W4A16_OK) return st;
  if ((st = check_ptr(workspace, 256, "workspace")) != W4A16_OK) return st;
  const Layout L = make_layout(*plan, num_tokens);
  return launch_prepare(*plan, L, nullptr, static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream),
                        logits, num_global, topk_ids, topk_weights);
}

w4a16_status w4a16_moe_set_stage_events(w4a16_moe_plan_t plan, void* const* events, int32_t n) {
  if (!plan) return fail(W4A16_ERR_INVALID_ARG, "plan is NULL");
  if (n == 0) {
    plan->has_ev = false;
    return W4A16_OK;
  }
  if (n != 4 || !events) return fail(W4A16_ERR_INVALID_ARG, "need exactly 4 events");
  for (int i = 0; i < 4; ++i) {
    if (!events[i]) return fail(W4A16_ERR_INVALID_ARG, "event %d is NULL", i);
    plan->ev[i] = static_cast<cudaEvent_t>(events[i]);
  }
  plan->has_ev = true;
  return W4A16_OK;
}

w4a16_status w4a16_moe_set_fused_finalize(w4a16_moe_plan_t plan, int32_t enable) {
  if (!plan) return fail(W4A16_ERR_INVALID_ARG, "plan is NULL");
  plan->finalize = enable != 0;
  return W4A16_OK;
}

w4a16_status w4a16_moe_set_weight_layout(w4a16_moe_plan_t plan, int32_t layout) {
  if (!plan) return fail(W4A16_ERR_INVALID_ARG, "plan is NULL");
  if (layout != W4A16_LAYOUT_CHECKPOINT && layout != W4A16_LAYOUT_INTERLEAVED)
    return fail(W4A16_ERR_INVALID_ARG, "unknown weight layout %d", layout);
  plan->layout = layout;
  return W4A16_OK;
}

w4a16_status w4a16_moe_relayout_weights(w4a16_moe_plan_t plan, int32_t which, const uint8_t* in, uint8_t* out,
                                        void* stream) {
  if (!plan) return fail(W4A16_ERR_INVALID_ARG, "plan is NULL");
  if (which != 0 && which != 1) return fail(W4A16_ERR_INVALID_ARG, "which must be 0 (W13) or 1 (W2), got %d", which);
  w4a16_status st;
  if ((st = check_ptr(in, 16, "in")) != W4A16_OK) return st;
  if ((st = check_ptr(out, 16, "out")) != W4A16_OK) return st;
  const w4a16_moe_desc& d = plan->d;
  const int32_t N = which == 0 ? (d.act == W4A16_ACT_SWIGLU ? 2 * d.inter : d.inter) : d.hidden;
  const int32_t K = which == 0 ? d.hidden : d.inter;
  const bool row_pairs = d.scale_kind == W4A16_SCALE_PER_CHANNEL;
  const size_t bytes = static_cast<size_t>(d.num_experts) * N * (K / 2);
  const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
  if (row_pairs && a < b + bytes && b < a + bytes)
    return fail(W4A16_ERR_INVALID_ARG, "per-channel relayout needs disjoint in / out buffers");
  if (!row_pairs && a != b && a < b + bytes && b < a + bytes)
    return fail(W4A16_ERR_INVALID_ARG, "in and out must be the same buffer or disjoint");
  cudaError_t e = launch_relayout(row_pairs, in, out, d.num_experts, N, K, plan->num_sms,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "relayout launch");
  return W4A16_OK;
}

const char* w4a16_moe_last_error(void) { return g_err.c_str(); }

}  // extern "C"

// ---------------------------------------------------------------------------
// Fixed-size workspace for callers that cannot allocate (see the header).
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) uint8_t g_static_workspace[W4A16_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_ws_mutex;
void* g_static_ws_ptr[kMaxDevices] = {nullptr};

// Device address of g_static_workspace on the current device (looked up once per
// device; the name is only a host-side stand-in for the device storage).
w4a16_status static_workspace_ptr(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(W4A16_ERR_UNSUPPORTED, "device index %d too large", dev);
  std::lock_guard<std::mutex> lock(g_static_ws_mutex);
  if (!g_static_ws_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_workspace);
    if (e != cudaSuccess || !ptr) return cuda_fail(e, "cudaGetSymbolAddress(static workspace)");
    g_static_ws_ptr[dev] = ptr;
  }
  *out = g_static_ws_ptr[dev];
  return W4A16_OK;
}

}  // namespace

extern "C" {

w4a16_status w4a16_moe_forward_static_workspace(w4a16_moe_plan_t plan, int32_t num_tokens, const void* x,
                                                const uint8_t* w13, const uint16_t* s13, const uint8_t* w2,
                                                const uint16_t* s2, const float* topk_weights,
                                                const int32_t* topk_ids, int32_t renormalize, void* out,
                                                void* stream) {
  if (!plan) return fail(W4A16_ERR_INVALID_ARG, "plan is NULL");
  if (num_tokens < 0 || num_tokens > plan->d.max_tokens)
    return fail(W4A16_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", num_tokens, plan->d.max_tokens);
  if (num_tokens == 0) return W4A16_OK;
  // device-side regions only: the host-call staging at the end of the layout
  // (from off_sx on) serves w4a16_moe_forward_host and the masked layout
  const size_t need = make_layout(*plan, num_tokens).off_sx;
  if (need > W4A16_STATIC_WORKSPACE_BYTES)
    return fail(W4A16_ERR_WORKSPACE_TOO_SMALL,
                "batch of %d tokens needs %zu bytes of workspace; the static workspace holds %u",
                num_tokens, need, W4A16_STATIC_WORKSPACE_BYTES);
  void* ws = nullptr;
  w4a16_status st = static_workspace_ptr(&ws);
  if (st != W4A16_OK) return st;
  st = w4a16_moe_prepare_routes(plan, num_tokens, topk_ids, ws, stream);
  if (st != W4A16_OK) return st;
  return w4a16_moe_forward(plan, num_tokens, x, w13, s13, w2, s2, topk_weights, topk_ids, renormalize, out,
                           ws, stream);
}

}  // extern "C"
