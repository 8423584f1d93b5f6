/*
 * w4a16_moe.h -- C ABI of the GB300 (sm_103a) local W4A16 MoE forward.
 *
 * The operation.  For T tokens with activations x[T, H], top-k expert ids and
 * FP32 routing weights, every valid route (t, j) to local expert e computes
 *
 *     h   = W13[e] . x[t]            gate/up GEMM, INT4 weights x 16-bit scales
 *     a   = silu(h_gate) * h_up      (SwiGLU)   or   a = max(h, 0)^2 (ReLU^2)
 *     y   = W2[e] . a                down GEMM
 *
 * and out[t] = cast( sum_{j = 0..k-1, route valid} w'[t, j] * y_{t,j} ), the
 * sum taken in FP32 in fixed top-k order with one final cast.  Sources:
 *   - "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy PR 4947),
 *     sections Modification and Benchmark: route preparation, gate/up GEMM,
 *     SiLU, down GEMM, weighted reduction; INT4 group size 32 with BF16
 *     scales; invalid routes and masked expert counts; split-K for small
 *     batches and route-count-based tile selection.
 *   - "perf: reduce split W4A16 routing and output overhead" (FlashInfer PR
 *     5186), section Description: expert outputs are stored in the 16-bit
 *     activation dtype, then combined in FP32 in fixed top-k order before one
 *     output cast, without atomics.
 *   - "[None][feat] Add W4A16 per-channel weight-only support for Cutlass
 *     fused MoE" (TensorRT-LLM PR 18313), sections Checkpoint format
 *     (per-output-channel scale = absmax/7, two INT4 per byte along the
 *     output dim, even index in the low nibble) and Validation (non-gated
 *     Relu2 arm).
 *
 * Conventions shared by all entry points
 *   - INT4 codes are two's complement nibbles in [-8, 7]; in every packed byte
 *     the even logical index sits in the low nibble.
 *   - Gated W13 holds the I gate rows first, then the I up rows.
 *   - Scales are always BF16.  Activations / output are BF16 or FP16.
 *   - Route validity: id != -1 and 0 <= id - expert_offset < num_experts.
 *     Other ids (routes that live on other ranks) are masked: they add
 *     nothing.  A token whose routes are all invalid gets an exact +0 row.
 *   - Sizes in the descriptor are LOGICAL (unpacked) sizes.  Packed sizes are
 *     derived from them; nothing is inferred from a pointer's element type.
 *   - Device pointers must be 16-byte aligned; arrays are dense row-major.
 *   - Calls are asynchronous on the given stream (a cudaStream_t passed as
 *     void*, NULL = legacy default stream).  prepare_routes and forward never
 *     allocate, synchronise or copy device->host, so both can be captured in a
 *     CUDA graph.
 *   - Errors are reported before any launch as a status code; the message of
 *     the most recent failing call on this host thread is returned by
 *     w4a16_moe_last_error().  Device-side work has no error conditions apart
 *     from a bounded-wait timeout inside the GEMM pipeline, which sets a flag
 *     in the workspace that w4a16_moe_check_device_error() reads.
 */
#ifndef W4A16_MOE_H
#define W4A16_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  W4A16_OK = 0,
  W4A16_ERR_INVALID_ARG = 1,       /* null / misaligned pointer, bad size */
  W4A16_ERR_UNSUPPORTED = 2,       /* shape or option the kernels do not cover */
  W4A16_ERR_WORKSPACE_TOO_SMALL = 3,
  W4A16_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed */
  W4A16_ERR_DEVICE_TIMEOUT = 5     /* a bounded wait inside a kernel gave up */
} w4a16_status;

typedef enum { W4A16_ACT_SWIGLU = 0, W4A16_ACT_RELU2 = 1 } w4a16_act;
typedef enum { W4A16_SCALE_GROUP32_K = 0, W4A16_SCALE_PER_CHANNEL = 1 } w4a16_scale;
typedef enum { W4A16_DT_BF16 = 0, W4A16_DT_FP16 = 1 } w4a16_dtype;
/* Packed weight layouts a forward can take (see w4a16_moe_relayout_weights). */
typedef enum {
  W4A16_LAYOUT_CHECKPOINT = 0,   /* the layouts documented with w4a16_moe_desc */
  W4A16_LAYOUT_INTERLEAVED = 1   /* the library's relaid-out layout */
} w4a16_weight_layout;
/* Where the two expert GEMMs run (see w4a16_moe_set_gemm_path). */
typedef enum {
  W4A16_PATH_AUTO = 0,          /* planner's choice per batch size */
  W4A16_PATH_TENSOR_CORES = 1,  /* tcgen05 MMA on dequantised tiles */
  W4A16_PATH_CUDA_CORES = 2     /* warp-MMA GEMV, route tiles of <= 8 routes */
} w4a16_gemm_path;

/*
 * Problem descriptor (logical sizes).
 *   num_experts   E, experts held by this GPU (1..1024)
 *   expert_offset global id of local expert 0 (>= 0); stands in for expert
 *                 parallelism: ids outside [offset, offset + E) are masked
 *   hidden        H, multiple of 32
 *   inter         I, multiple of 32
 *   top_k         k, 1..16
 *   max_tokens    largest T any later call may pass (1..65536)
 *   act           w4a16_act: SWIGLU (W13 has N1 = 2I rows) or RELU2 (N1 = I)
 *   scale_kind    w4a16_scale
 *   act_dtype     w4a16_dtype of x and out (and of the intermediate)
 *   global_experts experts the router spreads routes over (ids in [0, global_experts));
 *                 0 = num_experts.  Only the planner reads it: the expected routes per
 *                 local expert T * top_k / global_experts set the route-tile height and
 *                 the GEMM path.  Results do not depend on it.  0 or >= num_experts
 *                 (at most 1 << 20).
 *
 * Weight layouts (uint8 packed codes, uint16 BF16 scale bits):
 *   GROUP32_K:    W13 [E, N1, H/2]  S13 [E, N1, H/32]
 *                 W2  [E, H,  I/2]  S2  [E, H,  I/32]
 *                 byte b of a row holds K index 2b (low) and 2b+1 (high)
 *   PER_CHANNEL:  W13 [E, N1/2, H]  S13 [E, N1]
 *                 W2  [E, H/2,  I]  S2  [E, H]
 *                 byte [p, c] holds row 2p (low) and row 2p+1 (high)
 */
typedef struct {
  int32_t num_experts;
  int32_t expert_offset;
  int32_t hidden;
  int32_t inter;
  int32_t top_k;
  int32_t max_tokens;
  int32_t act;
  int32_t scale_kind;
  int32_t act_dtype;
  int32_t global_experts;
} w4a16_moe_desc;

typedef struct w4a16_moe_plan_s* w4a16_moe_plan_t;

/*
 * w4a16_moe_plan -- validate a descriptor and build a host-side plan.
 *   desc             problem descriptor (read only, copied)
 *   out              receives the plan handle (owned by the caller; free with
 *                    w4a16_moe_plan_destroy)
 *   workspace_bytes  receives the device workspace size that every later call
 *                    with num_tokens <= max_tokens needs
 * Host only: no device work, no allocation on the device.  Queries the current
 * device's SM count.  Returns INVALID_ARG / UNSUPPORTED for a bad descriptor.
 */
w4a16_status w4a16_moe_plan(const w4a16_moe_desc* desc, w4a16_moe_plan_t* out,
                            size_t* workspace_bytes);

/* Frees the plan's host memory.  NULL is accepted. */
w4a16_status w4a16_moe_plan_destroy(w4a16_moe_plan_t plan);

/*
 * w4a16_moe_prepare_routes -- route layout ("histogram") for one batch.
 * Passage: the LMDeploy page, Benchmark ("route preparation") and
 * Modification ("invalid routes and masked expert counts"); the FlashInfer
 * page, Description (top-k known at compile time in routing).
 *   num_tokens  T, 0 <= T <= max_tokens (T = 0: no-op)
 *   topk_ids    device int32 [T, k]
 *   workspace   device buffer of workspace_bytes (caller-owned); receives the
 *               per-expert counts, padded segment offsets, the stable
 *               slot -> route permutation, its inverse and the tile list
 *   stream      cudaStream_t as void*
 * Device result (read back with w4a16_moe_route_info offsets):
 *   counts[e]   valid routes of local expert e
 *   offs[e]     first slot of expert e; segments padded to the route-tile
 *               height bm; offs[E] = total slots
 *   perm[slot]  flat route t*k + j, -1 in padding slots; within an expert
 *               routes keep ascending flat order (stable)
 *   inv[r]      slot of route r, -1 when invalid or masked
 *   tiles[i]    int32 x4 (expert, first slot, valid rows, 0), i < num_tiles
 */
w4a16_status w4a16_moe_prepare_routes(w4a16_moe_plan_t plan, int32_t num_tokens,
                                      const int32_t* topk_ids, void* workspace, void* stream);

/*
 * w4a16_moe_forward -- gate/up GEMM + activation + down GEMM + FP32 top-k
 * combine, consuming the route layout that prepare_routes left in the same
 * workspace for the same topk_ids and num_tokens.
 * Passage: the LMDeploy page, Modification and Benchmark; the FlashInfer
 * page, Description (non-fused finalisation, FP32 fixed-order combine, one
 * cast, no atomics); the TensorRT-LLM page, Checkpoint format.
 *   x             device [T, H] act_dtype
 *   w13, s13      device packed gate/up (or fc1) weights and BF16 scales
 *   w2, s2        device packed down weights and BF16 scales
 *   topk_weights  device float32 [T, k]
 *   topk_ids      device int32 [T, k] (the ids given to prepare_routes)
 *   renormalize   nonzero: w'[t, j] = w[t, j] / sum_j w[t, j] (FP32, j
 *                 ascending, over all k entries; zero sum -> zero weights)
 *   out           device [T, H] act_dtype (written, never read)
 *   workspace     the buffer prepare_routes filled
 * All buffers are caller-owned.  Deterministic: identical inputs give
 * bit-identical outputs.
 */
w4a16_status w4a16_moe_forward(w4a16_moe_plan_t plan, int32_t num_tokens, const void* x,
                               const uint8_t* w13, const uint16_t* s13, const uint8_t* w2,
                               const uint16_t* s2, const float* topk_weights,
                               const int32_t* topk_ids, int32_t renormalize, void* out,
                               void* workspace, void* stream);

/*
 * w4a16_moe_forward_host -- end-to-end call with HOST activations, ids,
 * routing weights and output (expert weights stay resident on the device).
 * Copies x / ids / weights host->device into staging space inside the
 * workspace, runs prepare_routes + forward, and copies out back, all on
 * `stream`, then synchronises the stream.  Host buffers should be pinned for
 * asynchronous copies.  Same argument meaning as above otherwise.
 */
w4a16_status w4a16_moe_forward_host(w4a16_moe_plan_t plan, int32_t num_tokens, const void* x_host,
                                    const uint8_t* w13, const uint16_t* s13, const uint8_t* w2,
                                    const uint16_t* s2, const float* topk_weights_host,
                                    const int32_t* topk_ids_host, int32_t renormalize,
                                    void* out_host, void* workspace, void* stream);

/* Route-layout description for a batch of num_tokens (host only). */
typedef struct {
  int32_t tile_rows;       /* bm: route-tile height, also the MMA N */
  int32_t max_slots;       /* capacity of perm */
  int32_t max_tiles;       /* capacity of the tile list */
  int32_t gemm1_splits;    /* split-K factor of the gate/up GEMM */
  int32_t gemm2_splits;    /* split-K factor of the down GEMM */
  int32_t gemm1_ctas;      /* persistent grid sizes */
  int32_t gemm2_ctas;
  int32_t pipeline_stages; /* shared-memory stages of the gate/up GEMM ring */
  int32_t gemm_path;       /* W4A16_PATH_TENSOR_CORES or W4A16_PATH_CUDA_CORES */
  size_t off_counts, off_offs, off_perm, off_inv, off_tiles, off_num_tiles;  /* bytes */
  size_t off_inter;        /* intermediate activations [max_slots, I] (act dtype) */
  size_t off_expert_out;   /* expert outputs [max_slots, H] in the activation dtype, or FP32
                              split partials [gemm2_splits, max_slots, H] when gemm2_splits > 1 */
  int32_t fused_gemms;     /* 1: CUDA-core path with both GEMMs in one launch (then
                              gemm1_ctas = gemm2_ctas = that launch's grid: one CTA
                              per SM, or two with one compute group each) */
  int32_t fused_finalize;  /* 1: that launch also combines the routes (no combine launch) */
} w4a16_route_info;

w4a16_status w4a16_moe_route_info(w4a16_moe_plan_t plan, int32_t num_tokens,
                                  w4a16_route_info* info);

/*
 * Test / tuning overrides for later calls with this plan: force the route-tile
 * height (16..128, multiple of 16) and split-K factors (1..64; a factor larger
 * than the number of K blocks leaves empty partitions, which write zeros).
 * 0 restores the automatic choice.  workspace_bytes receives the workspace
 * size later calls need with these overrides in effect (it can exceed the
 * size plan reported).
 */
w4a16_status w4a16_moe_set_overrides(w4a16_moe_plan_t plan, int32_t tile_rows,
                                     int32_t gemm1_splits, int32_t gemm2_splits,
                                     size_t* workspace_bytes);

/*
 * Chooses where the expert GEMMs run for later calls with this plan.
 * W4A16_PATH_AUTO (the default) takes the CUDA-core GEMV while the expected
 * routes per local expert, num_tokens * top_k / num_experts, are at most 13
 * (group scales) or 10 (per-channel scales), or at most 80 when hidden and
 * inter are both at least 2048, and the tensor cores above that (measured
 * crossovers on GB300).  Both paths compute the same function
 * (the expert MLPs of "feat(pytorch): add CuTeDSL W4A16 MoE backend"
 * (LMDeploy), section Modification); they round differently (the tensor-core
 * path rounds each dequantised weight q * s to the activation type, the
 * CUDA-core path multiplies the exact codes q by the activations, sums a
 * 32-element group in FP32 and applies s to that sum), so outputs of the two
 * agree within the parity tolerance, not bit for bit.  The CUDA-core path
 * uses route tiles of 8, 16 or 32 routes (tile_rows overrides apply to the
 * tensor-core path only).  workspace_bytes (if not
 * NULL) receives the workspace size later calls need.  Unknown path:
 * W4A16_ERR_INVALID_ARG.
 */
w4a16_status w4a16_moe_set_gemm_path(w4a16_moe_plan_t plan, int32_t path, size_t* workspace_bytes);

/*
 * w4a16_moe_forward_masked -- the expert MLPs on the masked-count layout that a
 * low-latency expert-parallel dispatch hands over ("feat(pytorch): add CuTeDSL
 * W4A16 MoE backend" (LMDeploy), section Modification: invalid routes and
 * masked expert counts): x [num_experts, max_rows, H] act_dtype with counts[e]
 * valid rows for local expert e (rows past the count are ignored); y, same
 * shape, receives y[e][i] = W2[e] . act(W13[e] . x[e][i]) for i < counts[e]
 * and +0 rows elsewhere; the combine over top-k happens after the return
 * dispatch, outside this call.  Counts are clamped to [0, max_rows].  Every
 * row is one token with a single route of weight 1, so the plan must have
 * top_k == 1 and max_tokens >= num_experts * max_rows; prepare_routes and
 * forward run on that plan's workspace (the expanded routes live in its
 * staging area).  counts: device int32 [num_experts]; other arguments as for
 * w4a16_moe_forward.  max_rows == 0 is a no-op.  Errors: W4A16_ERR_UNSUPPORTED
 * (plan top_k != 1), W4A16_ERR_INVALID_ARG (negative max_rows, too many rows,
 * NULL/misaligned pointers), and those of prepare_routes / forward.
 */
w4a16_status w4a16_moe_forward_masked(w4a16_moe_plan_t plan, int32_t max_rows, const int32_t* counts,
                                      const void* x, const uint8_t* w13, const uint16_t* s13, const uint8_t* w2,
                                      const uint16_t* s2, void* y, void* workspace, void* stream);

/*
 * w4a16_moe_route_topk -- the router step before prepare_routes: softmax over
 * each token's router logits, then its top_k experts.  "feat(pytorch): add
 * CuTeDSL W4A16 MoE backend" (LMDeploy), section Benchmark, takes the routes
 * (INT32 expert ids, FP32 routing weights, renormalize=False) from a router
 * score / top-k computation.
 *   logits        [num_tokens, num_global] FP32, row-major (device, 4-byte
 *                 aligned); num_global = experts of the whole model, 1..1024
 *   top_k         1..min(16, num_global)
 *   topk_ids      [num_tokens, top_k] int32 out (device): global expert
 *                 indices by descending probability, ties to the lower index;
 *                 feed them (with the plan's expert_offset) to prepare_routes
 *                 and forward, which mask the experts of other ranks
 *   topk_weights  [num_tokens, top_k] FP32 out (device): the softmax
 *                 probabilities of the selected experts (not renormalised;
 *                 forward's `renormalize` does that)
 * The selection compares the logits exactly (softmax is increasing in them);
 * the probabilities are FP32.  Asynchronous on `stream`, no allocation, CUDA
 * graph capturable; num_tokens == 0 is a no-op.  Errors: W4A16_ERR_INVALID_ARG
 * (NULL or misaligned pointers, negative num_tokens), W4A16_ERR_UNSUPPORTED
 * (num_global or top_k out of range), W4A16_ERR_CUDA (launch failure).
 */
w4a16_status w4a16_moe_route_topk(const float* logits, int32_t num_tokens, int32_t num_global, int32_t top_k,
                                  int32_t* topk_ids, float* topk_weights, void* stream);

/*
 * w4a16_moe_route_and_prepare -- the router step and route preparation in one
 * pass: for every token, softmax over its router logits and its top_k experts
 * (exactly as w4a16_moe_route_topk), written to topk_ids / topk_weights, and
 * the route layout of those ids (exactly as w4a16_moe_prepare_routes) left in
 * the workspace for a following w4a16_moe_forward with the same ids and
 * weights.  The router's per-CTA expert counts feed the layout directly, so
 * the two steps take two kernels instead of three.  Passage: "feat(pytorch):
 * add CuTeDSL W4A16 MoE backend" (LMDeploy), section Benchmark (routes from a
 * router score / top-k step, then route preparation).
 *   logits        [num_tokens, num_global] FP32 (device); num_global = experts
 *                 of the whole model, 1..1024, >= the plan's top_k
 *   topk_ids      [num_tokens, top_k] int32 out (device, global ids)
 *   topk_weights  [num_tokens, top_k] FP32 out (device, softmax probabilities)
 *   workspace     the plan's workspace
 * Asynchronous on `stream`, no allocation, CUDA-graph capturable;
 * num_tokens == 0 is a no-op.  Errors: W4A16_ERR_INVALID_ARG (NULL or
 * misaligned pointers, num_tokens out of range), W4A16_ERR_UNSUPPORTED
 * (num_global out of range), W4A16_ERR_CUDA (launch failure).
 */
w4a16_status w4a16_moe_route_and_prepare(w4a16_moe_plan_t plan, int32_t num_tokens, const float* logits,
                                         int32_t num_global, int32_t* topk_ids, float* topk_weights, void* workspace,
                                         void* stream);

/*
 * w4a16_moe_relayout_weights -- plan-time relayout of one packed weight tensor
 * into W4A16_LAYOUT_INTERLEAVED, the order the GEMM kernels dequantise with
 * shifts and masks alone (no byte permutes).  Passages: "feat(pytorch): add
 * CuTeDSL W4A16 MoE backend" (LMDeploy), section Motivation (weights stay
 * packed INT4, no persistent BF16 expansion); "[None][feat] Add W4A16
 * per-channel weight-only support for Cutlass fused MoE" (TensorRT-LLM),
 * section Changes (setup-time preprocessing of the packed weights).  A
 * one-time setup step, outside any timed forward; codes are copied bit for
 * bit, the byte count does not change.
 *   which   0: W13 (N = N1 rows, K = hidden), 1: W2 (N = hidden rows, K = inter)
 *   in      device, the checkpoint layout of w4a16_moe_desc for the plan's
 *           scale_kind
 *   out     device, E x N x K/2 bytes: rows packed along K; in every 32-bit
 *           word (K values 8w .. 8w+7 of a row) the nibble at bit position 4p
 *           holds the code of K index 8w + {0,2,4,6,1,3,5,7}[p]
 *           GROUP32_K: out may equal in (in place) or be disjoint;
 *           PER_CHANNEL (row-pair input): out and in must be disjoint
 * Scales are not touched.  Later forwards read such weights after
 * w4a16_moe_set_weight_layout(plan, W4A16_LAYOUT_INTERLEAVED).  Asynchronous
 * on `stream`.  Errors: W4A16_ERR_INVALID_ARG (NULL / misaligned / overlapping
 * pointers, which not 0 or 1), W4A16_ERR_CUDA (launch failure).
 */
w4a16_status w4a16_moe_relayout_weights(w4a16_moe_plan_t plan, int32_t which, const uint8_t* in, uint8_t* out,
                                        void* stream);

/*
 * Declares the layout of the packed weights that later forward calls on this
 * plan receive (both W13 and W2): W4A16_LAYOUT_CHECKPOINT (the default) or
 * W4A16_LAYOUT_INTERLEAVED (the output of w4a16_moe_relayout_weights).  Both
 * layouts give bit-identical results.  Host only; unknown layout:
 * W4A16_ERR_INVALID_ARG.
 */
w4a16_status w4a16_moe_set_weight_layout(w4a16_moe_plan_t plan, int32_t layout);

/*
 * Deterministic fused finalize ("perf: reduce split W4A16 routing and output
 * overhead" (FlashInfer), sections Description and Benchmarks: the combine
 * done inside the down GEMM's epilogue instead of a separate pass).  With
 * enable != 0, forwards that take the CUDA-core path with both GEMMs in one
 * launch (w4a16_route_info.fused_gemms) combine the routes there: no data
 * atomics -- per (token, 16-column block) arrival counters elect the warp of
 * the token's last valid route, which sums the token's expert outputs in
 * top-k order with the combine's arithmetic.  The output is bit-identical to
 * the separate combine after the same expert GEMMs: the fused finalize runs
 * the launch with two compute groups per CTA, so it equals a combine-launch
 * forward of that form (W4A16_MOE_FUSED_GROUPS=2); where the planner gives
 * the combine-launch forward one group per CTA, the two differ only in the
 * FP32 summation order of the units' K stages.  Other forwards are unaffected.  Default: off (also
 * set by the environment variable W4A16_MOE_FUSED_FINALIZE=1 at plan
 * creation).  Host only; plan NULL: W4A16_ERR_INVALID_ARG.
 */
w4a16_status w4a16_moe_set_fused_finalize(w4a16_moe_plan_t plan, int32_t enable);

/*
 * Reads (synchronously, on `stream`) and clears the device error flag in the
 * workspace.  Returns W4A16_ERR_DEVICE_TIMEOUT if a kernel gave up waiting
 * since the last prepare_routes on this workspace (prepare_routes clears it).
 * workspace == NULL reads the fixed workspace of
 * w4a16_moe_forward_static_workspace on the current device.
 * Every bounded wait in the GEMM pipelines gives up after 2 s by default; the
 * environment variable W4A16_MOE_WAIT_TIMEOUT_NS, read when a plan is created,
 * sets a different limit in nanoseconds for that plan's forwards (a test hook:
 * a limit shorter than a normal wait makes the kernels give up, wind down
 * their copies and MMAs and return, and this call then reports the timeout).
 */
w4a16_status w4a16_moe_check_device_error(w4a16_moe_plan_t plan, void* workspace, void* stream);

/*
 * Diagnostic timing hook.  With n == 4 and non-NULL `events` (cudaEvent_t
 * handles passed as void*), later forward calls on this plan record
 * events[0] before the gate/up GEMM, events[1] after it, events[2] after the
 * down GEMM and events[3] after the combine, on the forward's stream.  The
 * recordings separate the kernels, so the programmatic-launch overlap between
 * them is lost while they are on.  n == 0 turns the hook off.  The plan does
 * not own the events.
 */
w4a16_status w4a16_moe_set_stage_events(w4a16_moe_plan_t plan, void* const* events, int32_t n);

/*
 * w4a16_moe_forward_static_workspace -- prepare_routes + forward without any
 * caller-provided workspace and without allocating anything.
 * No counterpart on the pages: this is a library convenience for callers that
 * cannot allocate device memory themselves -- for instance code that runs
 * inside a CUDA graph capture (where cudaMalloc is not allowed), applications
 * whose memory is reserved up front by a pool that libraries may not bypass,
 * or plug-in hosts that give a library no allocator.
 *   The scratch lives in one file-scope device array of
 *   W4A16_STATIC_WORKSPACE_BYTES (32 MiB), which every GPU that loads this
 *   library holds until the process exits.  Batches whose layout needs more
 *   return W4A16_ERR_WORKSPACE_TOO_SMALL before any launch (the regular entry
 *   points report the need as workspace_bytes / w4a16_route_info).
 *   The first call on a device (with that device current) looks up the
 *   array's device address; make that first call before any stream capture.
 *   Every call shares the one array and leaves its contents behind (route
 *   preparation clears what must start at zero), so calls that overlap on the
 *   GPU -- on different streams without ordering -- race and must be avoided.
 *   w4a16_moe_check_device_error(plan, NULL, stream) reads this array's
 *   timeout flag.
 *   No cudaMalloc, cudaFree or allocating library routine is called.
 * Arguments as for w4a16_moe_forward (device pointers, same layouts).
 */
#define W4A16_STATIC_WORKSPACE_BYTES (32u * 1024u * 1024u)
w4a16_status w4a16_moe_forward_static_workspace(w4a16_moe_plan_t plan, int32_t num_tokens,
                                                const void* x, const uint8_t* w13,
                                                const uint16_t* s13, const uint8_t* w2,
                                                const uint16_t* s2, const float* topk_weights,
                                                const int32_t* topk_ids, int32_t renormalize,
                                                void* out, void* stream);

/* Message for the last non-OK status on this host thread ("" if none). */
const char* w4a16_moe_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_MOE_H */
