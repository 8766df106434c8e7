/*
 * moe_gb300.h -- C ABI of the dropless routed-expert MoE layer on one GB300.
 *
 * One GPU holds all E experts (no expert parallelism, no peer buffers).  The
 * caller supplies top-K expert IDs and scores per token; the library routes
 * and permutes the token rows by expert, runs a grouped W13 (gate + up) GEMM
 * with a fused SwiGLU epilogue and a grouped W2 GEMM on the tcgen05 tensor
 * cores, and sums each token's K score-weighted expert outputs in a fixed
 * order.  The backward pass produces dX, dW13 and dW2.
 *
 * Sources (page title, section):
 *   [DM]   "Dist-MoE: Speed-of-light distributed Mixture-of-Experts kernels",
 *          visual explainer (meta-pytorch.org/dist_moe).
 *   [BLOG] "Mixture of Experts: How Routing Becomes GPU Computation"
 *          (g-u-n.github.io).
 *   [NEWS] "Meta Dist-MoE: Open-Source Fused MoE Kernels for Blackwell"
 *          (explainx.ai).
 *
 * Conventions that hold for every call below
 *   - All tensors are row-major and contiguous; device pointers unless a
 *     parameter says "host".  Every device pointer must be 16-byte aligned.
 *   - Calls that take a cudaStream_t only enqueue work on that stream.  They
 *     never allocate, never synchronise and never read device memory on the
 *     host, so a sequence of them can be captured in a CUDA graph; the
 *     addresses the context owns never change after moe_ctx_create.
 *   - Host-detectable errors (NULL pointers, sizes above the context's
 *     capacity, shape or precision mismatches, misaligned pointers) return a
 *     status synchronously and enqueue nothing.
 *   - Errors the GPU detects (IDs outside [-1, E), an ID of -1 carrying a
 *     nonzero score when MOE_DEBUG_CHECKS is set, a device wait that ran out
 *     of time) never trap: the kernel sets a bit in the context's error word
 *     and carries on (a bad ID is treated as inactive).  moe_ctx_get_error
 *     reads and clears the word.
 *   - A context is reusable sequentially but not reentrant: calls that may
 *     overlap on the GPU need separate contexts ([DM] section 04, last
 *     paragraph of "Save and Recompute Decisions"; [NEWS] "How the execution
 *     model works").
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* NULL/misaligned pointer, bad size or shape */
  MOE_ERR_CAPACITY = 2,      /* T above the context's max_tokens           */
  MOE_ERR_BAD_ROUTE = 3,     /* reserved: routes are checked on the GPU    */
  MOE_ERR_UNSUPPORTED = 4,   /* shape the kernels do not tile (see below)  */
  MOE_ERR_CUDA = 5,          /* a CUDA runtime call failed                 */
  MOE_ERR_TIMEOUT = 6        /* reserved: device timeouts set an error bit */
} moe_status;

/* Bits of the device error word (moe_ctx_get_error). */
#define MOE_DEV_ERR_BAD_ID          0x1u  /* an ID outside [-1, E) was seen     */
#define MOE_DEV_ERR_INACTIVE_SCORE  0x2u  /* ID -1 with score != 0 (debug only) */
#define MOE_DEV_ERR_TIMEOUT         0x4u  /* a bounded device wait expired      */

/* MOE_MXFP8_1X32 is a weight preparation, not a layer precision: MXFP8
 * weights with one scale per 1x32 block along K ("Meta Dist-MoE:
 * Open-Source Fused MoE Kernels for Blackwell", "Supported modes": 32x32
 * blocks for training-compatible values, 1x32 for inference).  Such a
 * weight feeds moe_forward of an MXFP8 context; moe_backward rejects it. */
/* MOE_NVFP4 is an inference precision ([DM] section 02, "Expert
 * Computation and Tensor Precision": E2M1 values with E4M3 block scales and
 * a global scale per row; section 08, "Public API and Supported Modes":
 * NVFP4 inference with prepared weights): a context of this precision takes
 * no MOE_TRAINING, MOE_REPLAY or MOE_POST_NORM flag (MOE_ERR_UNSUPPORTED)
 * and its moe_forward runs without `saved` and without MOE_FUSED_LAUNCH.
 * Weights, x rows and h2 rows are quantised along K in blocks of 16 values:
 * g = amax(row) / 2688, sb = E4M3(amax(block) / (6 g)), q = E2M1(v / (sb g)),
 * each step one FP32 operation rounded to nearest even (E4M3 and E2M1
 * saturate); h1 and h3 are rounded to BF16 as in the other precisions. */
typedef enum { MOE_BF16 = 0, MOE_MXFP8 = 1, MOE_MXFP8_1X32 = 2, MOE_NVFP4 = 3 } moe_precision;

/* moe_config.flags */
#define MOE_TRAINING      0x1u  /* forward saves state; backward is allowed   */
#define MOE_DEBUG_CHECKS  0x2u  /* also flag ID -1 routes with nonzero score */
#define MOE_POST_NORM     0x4u  /* the layer ends with the post-expert RMSNorm
                                   (moe_ctx_set_post_norm); training saves the
                                   pre-norm output for moe_post_norm_backward */
#define MOE_REPLAY        0x8u  /* (with MOE_TRAINING) the context also holds
                                   the scratch a backward uses to rebuild the
                                   expert state of a forward that saved only
                                   its input (MOE_SAVE_INPUT_ONLY); see
                                   "Activation slots" below                 */

/* call_flags of moe_forward */
#define MOE_ACCUMULATE_OUT 0x1u /* out = round(out + sum_k s*h3) (shared expert first) */
#define MOE_FUSED_LAUNCH   0x4u /* inference, MXFP8: the whole forward in one
                                   launch (see moe_forward)                    */
#define MOE_SAVE_INPUT_ONLY 0x2u /* training: `saved` is an input-only state of
                                    moe_saved_input_bytes (routing, scores, a
                                    copy of x); needs a MOE_REPLAY context    */
/* call_flags of moe_backward */
#define MOE_ACCUMULATE_DX  0x1u /* dx  = round(dx + sum_k dxr)                 */
#define MOE_DW_FP32        0x2u /* dW13/dW2 are float32 instead of BF16        */
#define MOE_DW_ACCUMULATE  0x4u /* dW += new gradient (in the dW dtype)        */
#define MOE_REPLAY_FORWARD 0x8u /* `saved` was written with MOE_SAVE_INPUT_ONLY:
                                   rebuild the expert state first (must match
                                   the forward's choice)                      */

/*
 * Layer shape and precision.  The kernels tile D and F in steps of 128, so
 * d_model % 128 == 0 and d_ff % 128 == 0 are required (MOE_ERR_UNSUPPORTED
 * otherwise); num_experts <= 1024, top_k <= 32.
 *   BF16:  BF16 operands, FP32 accumulation, BF16 stored intermediates.
 *   MXFP8: E4M3 operands with one E8M0 scale per 32 values along the
 *          contraction axis ([DM] section 02, "Block-Scaled Quantization"),
 *          FP32 accumulation, BF16 h1/h3.
 *   NVFP4: (inference) E2M1 operands with E4M3 scales per 16 values and an
 *          FP32 scale per row (see moe_precision), FP32 accumulation of the
 *          scaled codes, BF16 h1/h3; h2 formed in FP32, then quantised.
 */
typedef struct {
  int32_t max_tokens;     /* T_max: largest T any call will pass            */
  int32_t d_model;        /* D                                              */
  int32_t d_ff;           /* F (h1 has 2F columns: gate then up)            */
  int32_t num_experts;    /* E                                              */
  int32_t top_k;          /* K routes per token                             */
  moe_precision precision; /* MOE_BF16, MOE_MXFP8 or MOE_NVFP4 (inference)  */
  uint32_t flags;         /* MOE_TRAINING | MOE_DEBUG_CHECKS                */
  float swiglu_limit;     /* 0: plain SwiGLU.  L > 0: clamped SwiGLU ("Meta
                           * Dist-MoE...", "Supported modes"), h2 =
                           * SiLU(min(g, L)) * clamp(u, -L, L) on the BF16 h1;
                           * the backward's gradient is zero where g > L
                           * (for g) or |u| > L (for u).  Finite, >= 0.   */
} moe_config;

/*
 * One stacked expert weight [E, N, K] (K contiguous) as the GEMMs read it.
 *   W13: N = 2F, K = D (rows 0..F-1 gate, F..2F-1 up; [DM] section 01
 *        "Inputs, shapes, and inactive routes", [BLOG] section 2
 *        grouped_swiglu_forward_combined).
 *   W2:  N = D,  K = F.
 * BF16:  data = the caller's BF16 tensor; scale = scale_t = NULL; data_t =
 *        BF16 [E, K, N] transposed copy (needed by moe_backward only).
 * MXFP8: data = E4M3 codes [E, N, K], scale = E8M0 atoms [E*N/128][K/128];
 *        scale_t = E8M0 atoms [E*K/128][N/128] (backward only), and
 *        optionally data_t = E4M3 codes [E, K, N] (backward only).  With
 *        data_t == NULL the input-gradient GEMMs read `data` itself,
 *        MN-major ([DM] section 02, "Quantization Axes for Forward and
 *        Backward": static 32x32 weights let FPROP and DGRAD share qdata),
 *        which saves E*N*K bytes; with data_t they read the K-major copy.
 *        Both give the same results.  Atoms: E*N*K/32 bytes, see below.
 *        N % 128 == 0 and K % 128 == 0.  Filled by prepare_block_scaled_weight.
 * NVFP4: data = chunks of 128 rows x 64 values (4096 bytes of E2M1 codes, row
 *        m at byte 32 m, value k in byte k/2, low nibble for even k; then
 *        512 bytes of E4M3 block scales, row m's four at 4096 + 4 m), the
 *        chunk of rows 128 t .. 128 t + 127 of the stacked [E*N, K] weight
 *        and values 64 s .. 64 s + 63 at (t * K/64 + s) * 4608;
 *        scale = FP32 row scales g [E*N]; data_t = scale_t = NULL.
 * The struct is read on the host at call time; the pointers are not owned.
 */
typedef struct {
  moe_precision precision;
  int32_t E, N, K;
  const void* data;
  const uint8_t* scale;
  const void* data_t;
  const uint8_t* scale_t;
} moe_weight;

typedef struct moe_ctx moe_ctx;

/*
 * Create a context: checks the config, allocates all scratch once (every
 * later call reuses it, so its addresses are stable for graph capture) and
 * creates no stream.  Scratch is sized for max_tokens*top_k routes plus 31
 * pad rows per expert, which bounds every routing, so a call can never
 * overflow it ([NEWS] "How the execution model works" treats running out of
 * scratch as fatal; here it is sized so that cannot happen).  Must be called with the target device current.
 * Returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_CUDA; *out is
 * set only on MOE_OK.
 */
MOE_API moe_status moe_ctx_create(const moe_config* cfg, moe_ctx** out);

/* Free the context's scratch.  The caller must make sure no enqueued work
 * that uses it is still running (synchronise first). */
MOE_API moe_status moe_ctx_destroy(moe_ctx* ctx);

/* Bytes of device scratch a context with this config allocates (0 if the
 * config is invalid). */
MOE_API size_t moe_ctx_scratch_bytes(const moe_config* cfg);

/*
 * Bytes of the per-layer saved state that a training forward writes and the
 * matching backward reads: routing arrays, a copy of the scores, BF16 h1
 * [R_cap, 2F], the WGRAD column bundles of x and h2 and BF16 h3 [R_cap, D]
 * ([DM] section 04, "Activation Lifetimes and Backward Readers": MXFP8
 * full-save keeps the x/h2 column bundles, dense h1 and h3).  The caller allocates it (16-byte aligned)
 * and keeps one per live layer.  0 for an invalid config.
 */
MOE_API size_t moe_saved_state_bytes(const moe_config* cfg);

/*
 * Layout of every MXFP8 scale array (weights, row bundles, column bundles):
 * 512-byte atoms, each holding the E8M0 scales of 128 operand rows x 4
 * consecutive 32-value blocks along the contraction axis.  Row p (0..127) of
 * the atom and block l (0..3) sit at byte (p % 32) * 16 + (p / 32) * 4 + l,
 * the order in which tcgen05.cp 32x128b.warpx4 lays a row's scales into
 * tensor memory, so a GEMM stage moves its scales with one bulk copy.
 *   weight scale    atoms [E*N/128][K/128]   (rows = weight rows)
 *   weight scale_t  atoms [E*K/128][N/128]
 *   row bundles     atoms [B_cap][Kdim/128]  (rows = rows of routing block b,
 *                   counted from the block's first row)
 *   column bundles  atoms [Dim/128][B_cap]   (rows = features; block l = the
 *                   32-row group l of routing block b)
 * B_cap = (max_tokens*top_k + 31*E)/128 + E + 1 row blocks.
 */

/* Saved-state fields, for inspection by tests (moe_saved_state_field,
 * moe_saved_input_field).  The routing fields come first in memory
 * (HEADER..SCORES, BSTART, ROWBLOCK), then PRENORM, then H1, the column
 * bundles and H3 of a full state or X of an input-only state.  The routing
 * fields and PRENORM sit at the same offsets in both layouts. */
typedef enum {
  MOE_SAVED_HEADER = 0,     /* int32[16]: [0] T, [1] row blocks, [2] rows used, [3] active routes,
                               [4] row-block pairs                             */
  MOE_SAVED_COUNTS = 1,     /* int32[E]     active routes per expert           */
  MOE_SAVED_OFFSETS = 2,    /* int32[E+1]   exclusive prefix of counts         */
  MOE_SAVED_POFFSETS = 3,   /* int32[E+1]   same with counts padded to 32      */
  MOE_SAVED_PERM = 4,       /* int32[R_cap] route t*K+k of each row, -1 = pad  */
  MOE_SAVED_INV = 5,        /* int32[T_max*K] row of each route, -1 = inactive */
  MOE_SAVED_BLOCKS = 6,     /* int32[4*B_cap] (expert, first row, rows, pair):
                               each expert's padded rows cut into blocks of
                               <=128.  Word 3 of entry p < header[4] describes
                               row-block pair p, consecutive blocks of one
                               expert taken two at a time (the last alone):
                               (first block << 1) | (second block present);
                               0 in the other entries                          */
  MOE_SAVED_SCORES = 7,     /* float[T_max*K] scores, 0 for inactive routes    */
  MOE_SAVED_H1 = 8,         /* bf16[R_cap, 2F]                                 */
  MOE_SAVED_XCOL = 9,       /* x column bundle: bf16 [D, R_cap] or e4m3 codes  */
  MOE_SAVED_XCOL_SCALE = 10,/* e8m0 column-bundle atoms [D/128][B_cap] (MXFP8) */
  MOE_SAVED_H2COL = 11,     /* h2 column bundle: bf16 [F, R_cap] or e4m3       */
  MOE_SAVED_H2COL_SCALE = 12,/* e8m0 column-bundle atoms [F/128][B_cap]        */
  MOE_SAVED_BSTART = 13,    /* int32[E+1]   first row block of each expert     */
  MOE_SAVED_ROWBLOCK = 14,  /* int32[R_cap/32] row block of each 32-row group  */
  MOE_SAVED_H3 = 15,        /* bf16[R_cap, D] route outputs (score gradient)   */
  MOE_SAVED_PRENORM = 16,   /* bf16[T_max, D] layer output before the post-expert
                               RMSNorm (MOE_POST_NORM only, else 0 bytes)     */
  MOE_SAVED_X = 17,         /* bf16[T_max, D] the layer input x (input-only
                               states; 0 bytes in a full state)               */
  MOE_SAVED_NUM_FIELDS = 18
} moe_saved_field;

/* Offset and size in bytes of one saved-state field; the row capacity
 * R_cap used by the layouts above is returned by moe_row_capacity. */
MOE_API moe_status moe_saved_state_field(const moe_config* cfg, int field, size_t* offset, size_t* bytes);

/* R_cap: rows of every per-route buffer = max_tokens*top_k + 31*E rounded
 * up to a multiple of 128, plus 128 (0 for an invalid config). */
MOE_API int64_t moe_row_capacity(const moe_config* cfg);

/*
 * Prepare one stacked expert weight once, outside any timed region
 * ([NEWS] "Supported modes": prepare_block_scaled_weight quantises expert
 * weights once with 32x32 blocks for MXFP8 training; [DM] section 02: with
 * 32x32 blocks the forward and input-gradient GEMMs share qdata with
 * distinct scale orientations).
 *   w       BF16 [E, N, K] (device).  N % 32 == 0 and K % 32 == 0 (BF16),
 *           N % 128 == 0 and K % 128 == 0 (MXFP8).
 *   MXFP8:  one E8M0 scale per 32x32 tile (OCP MX rule: floor(log2 amax) - 8,
 *           values rounded to nearest-even E4M3 and saturated at 448) is
 *           written to the scale atoms [E*N/128][K/128] and, when
 *           scale_t != NULL, the input-gradient orientation's atoms
 *           [E*K/128][N/128]; if data_t != NULL too, the transposed codes
 *           [E,K,N] (data_t without scale_t is rejected).  data may not be
 *           NULL.
 *   MXFP8_1X32: inference weights, one E8M0 scale per 32 consecutive values
 *           of a row along K (same rule), codes to data [E,N,K] and scales
 *           to the atoms [E*N/128][K/128]; data_t and scale_t must be NULL.
 *           Use the result with moe_weight.precision = MOE_MXFP8_1X32.
 *   BF16:   data and scale must be NULL; data_t (BF16 [E,K,N]) receives the
 *           transpose used by the input-gradient GEMMs.
 *   NVFP4:  inference weights (the quantiser of MOE_NVFP4, blocks of 16
 *           along K, one row scale per weight row): codes and block scales
 *           to data, FP32 row scales to scale (see moe_weight); data_t and
 *           scale_t must be NULL; N % 128 == 0 and K % 64 == 0.
 * The outputs are caller-owned device buffers.  Enqueued on `stream`.
 */
/*
 * Bytes of the buffers prepare_block_scaled_weight fills for one [E, N, K]
 * weight, written to bytes[0..3] = data, scale, data_t, scale_t (0 for a
 * buffer the precision does not use).  `with_transpose` asks for the
 * backward's orientation (not for MOE_MXFP8_1X32): 0 none, 1 the transposed
 * codes and their scales, 2 (MXFP8) the scales only, for MN-major
 * input-gradient GEMMs that read the forward codes.
 *   MXFP8, MXFP8_1X32: data E*N*K, scale E*N*K/32 + 16, data_t E*K*N
 *                      (with_transpose 1), scale_t E*K*N/32 + 16 (1 or 2;
 *                      16 bytes of slack after the atoms); N % 128 == 0
 *                      and K % 128 == 0.
 *   BF16:              data E*N*K*2 (the caller's own tensor, which the
 *                      layer reads in place), data_t E*K*N*2.
 *   NVFP4:             data E*N*K*9/16 (codes and block scales), scale
 *                      E*N*4 (row scales); N % 128 == 0, K % 64 == 0,
 *                      with_transpose 0.
 * Host-only, no CUDA call.  Errors: MOE_ERR_INVALID_ARG (null bytes, shapes
 * prepare_block_scaled_weight rejects, with_transpose for MXFP8_1X32).
 */
MOE_API moe_status moe_weight_bytes(moe_precision precision, int32_t E, int32_t N, int32_t K, int with_transpose,
                                    size_t* bytes);

MOE_API moe_status prepare_block_scaled_weight(const void* w, int32_t E, int32_t N, int32_t K,
                                       moe_precision precision, void* data, uint8_t* scale,
                                       void* data_t, uint8_t* scale_t, cudaStream_t stream);

/*
 * Forward of the routed layer ([BLOG] section 2 "SwiGLU forward: compute
 * and combine expert outputs"; [DM] sections 01-02):
 *   x          bf16 [T, D]
 *   topk_ids   int32 [T, K]  expert of each route; -1 marks an inactive route
 *   topk_scores float [T, K] route weight; an inactive route's score is ignored
 *   W13, W2    prepared weights of the context's precision (see moe_weight)
 *   out        bf16 [T, D]   out[t] = bf16(sum_k s*h3), summed in FP32 in
 *                            k order; a token with no active route gets 0.
 *                            With MOE_ACCUMULATE_OUT the old out is added
 *                            first (one rounding at the end).
 *   saved      NULL for inference; for a training context, a buffer of
 *              moe_saved_state_bytes that the matching moe_backward reads.
 *              With MOE_SAVE_INPUT_ONLY (MOE_REPLAY context) a buffer of
 *              moe_saved_input_bytes instead: the forward keeps its routing,
 *              scores and a copy of x there and nothing of the expert
 *              state, which the backward rebuilds.
 * T may be 0 (nothing is enqueued).  T > max_tokens gives MOE_ERR_CAPACITY.
 *
 * MOE_NVFP4 contexts: inference only (saved must be NULL), NVFP4 weights;
 * the x rows are quantised into the routing blocks' chunks, the W13 +
 * SwiGLU GEMM writes FP32 h2, whose rows are quantised in turn, and the W2
 * GEMM writes BF16 h3 (six launches).
 *
 * MOE_FUSED_LAUNCH ([DM] section 05, "Kernel Pipelines: Staged and Mega":
 * the Mega forward joins W13 and W2 in one grid with readiness counters):
 * the routing, gather, W13 + SwiGLU GEMM, W2 GEMM and combine run as one
 * persistent cooperative launch (at most one CTA per SM) whose CTAs wait on
 * counters in the context's scratch for the records they consume; a
 * decode-sized step pays one launch instead of five, and the W2 weights
 * stream while W13 runs.  The result equals the staged forward's bit for
 * bit.  Inference only (saved == NULL), MXFP8 contexts, d_model % 256 == 0,
 * T*top_k <= 1024 and T*top_k/128 + min(num_experts, T*top_k) < 1024;
 * otherwise MOE_ERR_UNSUPPORTED (MOE_POST_NORM too).  A wait that runs past
 * its deadline sets MOE_DEV_ERR_TIMEOUT and the kernel returns; the
 * context stays usable.  Stage timing records one stage (the whole launch).
 */
MOE_API moe_status moe_forward(moe_ctx* ctx, int32_t T, const void* x, const int32_t* topk_ids,
                       const float* topk_scores, const moe_weight* W13, const moe_weight* W2,
                       void* out, void* saved, uint32_t call_flags, cudaStream_t stream);

/*
 * Backward of the routed layer ([BLOG] section 2 "SwiGLU backward: the
 * complete expert path"; [DM] section 05 "Kernel Pipelines": W2 DGRAD and
 * WGRAD, then SwiGLU backward with row and column grad_h1, then W13 DGRAD and
 * WGRAD, then the K-reduction of the input gradients):
 *   saved   the state written by the matching training forward
 *   dout    bf16 [T, D]   gradient of out (T as in that forward)
 *   W13,W2  prepared weights with the backward orientation: data_t (BF16);
 *           scale_t, with or without data_t (MXFP8)
 *   dx      bf16 [T, D]   dx[t] = bf16(sum_k dxr); MOE_ACCUMULATE_DX adds the
 *                         old dx first
 *   dW13    [E, 2F, D], dW2 [E, D, F]: BF16, or float with MOE_DW_FP32;
 *           MOE_DW_ACCUMULATE adds into them.  An expert no active route
 *           reaches gets exact zeros (or is left as is when accumulating).
 *   d_scores float [T, K] or NULL: the score gradient
 *           dp(t,k) = <h3(t,k), dout[t]> summed in FP32 in a fixed order
 *           ([BLOG] section 2 "SwiGLU backward": the routing-weight gradient
 *           of the weighted combine, which the caller's router backward
 *           consumes); 0 for inactive routes.
 *   MOE_REPLAY_FORWARD: `saved` is an input-only state.  Before the steps
 *           above the backward replays the forward's gather and W13 +
 *           SwiGLU GEMM (and its W2 GEMM when d_scores is requested) on the
 *           saved x and routing, writing the state into the context's
 *           MOE_BUF_REPLAY scratch, and reads it from there.  The replayed
 *           kernels and inputs are the forward's, so the gradients equal
 *           those of a full-state backward bit for bit.  The flag must
 *           match the forward's MOE_SAVE_INPUT_ONLY (moe_slot keeps it): the
 *           context remembers, per `saved` pointer, the last of its
 *           forwards that wrote there (up to 4096 pointers; past that it
 *           starts over), and a mismatch returns MOE_ERR_INVALID_ARG.
 */
MOE_API moe_status moe_backward(moe_ctx* ctx, const void* saved, const void* dout,
                        const moe_weight* W13, const moe_weight* W2, void* dx, void* dW13,
                        void* dW2, float* d_scores, uint32_t call_flags, cudaStream_t stream);

/* Synchronise the device, return the error word's bits in *bits and clear
 * it.  Not for use inside graph capture. */
MOE_API moe_status moe_ctx_get_error(moe_ctx* ctx, uint32_t* bits);

/* Clip statistics of the clamped SwiGLU ("Meta Dist-MoE: Open-Source Fused
 * MoE Kernels for Blackwell", "Supported modes" lists clip statistics; the
 * page does not define them, so these are the counts of the clamp): the
 * numbers of gate values above swiglu_limit (counts[0]) and of up values
 * outside [-limit, limit] (counts[1]) that every moe_forward since the last
 * call of this function clamped, over routed rows (pad rows never clip).
 * Zero with swiglu_limit == 0.  Synchronises the device, then clears the
 * counters.  Not for use inside graph capture. */
MOE_API moe_status moe_ctx_clip_stats(moe_ctx* ctx, uint64_t* counts);

/*
 * Stage timing, for measurement.  When enabled, moe_forward and moe_backward
 * record a CUDA event on their stream before their first launch and after
 * each stage (inside stream capture the records become event nodes of the
 * graph, so replays re-time them).  moe_ctx_stage_times waits for the events
 * of the last forward (pass 0) or backward (pass 1) and returns each stage's
 * duration in milliseconds:
 *   forward  (MOE_FWD_STAGES): route, gather x (row bundle, and the column
 *            bundle in the same pass when training), W13 + SwiGLU GEMM, W2
 *            GEMM, combine
 *   backward (MOE_BWD_STAGES): gather dh3 (row and column bundles), W2 DGRAD
 *            + SwiGLU backward GEMM, W2 WGRAD GEMM, W13 DGRAD GEMM, W13 WGRAD
 *            GEMM, dX reduction
 * The first enable creates the events (call it outside capture); they live
 * until moe_ctx_destroy, so disabling only stops later calls from recording
 * and a graph captured with timing on can still be replayed and read.
 * Destroy the context only after the last replay of such a graph.
 */
#define MOE_FWD_STAGES 5
#define MOE_BWD_STAGES 6
MOE_API moe_status moe_ctx_enable_stage_timing(moe_ctx* ctx, int enable);
MOE_API moe_status moe_ctx_stage_times(moe_ctx* ctx, int pass, float* ms, int n);

/*
 * Post-expert RMSNorm ("Meta Dist-MoE: Open-Source Fused MoE Kernels for
 * Blackwell", "Supported modes", names a fused post-expert RMSNorm without
 * defining it; this library's reading).  With MOE_POST_NORM in the
 * configuration, the combine that writes the layer output x[t] (the BF16
 * row of the score-weighted K-sum, after adding `out` under
 * MOE_ACCUMULATE_OUT) normalises it over D in the same pass:
 *   r[t] = 1 / sqrt(mean_d x[t,d]^2 + eps),  out[t,d] = bf16(gamma[d] x[t,d] r[t])
 * with r and the products in FP32.  A training forward also writes x to the
 * saved field MOE_SAVED_PRENORM.
 *
 * moe_ctx_set_post_norm: gamma is a device pointer to bf16[D] (16-byte
 *   aligned, not owned, read by every later forward and post-norm backward;
 *   keep it alive and unchanged while they run); eps finite and > 0.  A
 *   forward with MOE_POST_NORM and no gamma set returns MOE_ERR_INVALID_ARG.
 *   Errors: MOE_ERR_INVALID_ARG (null context or gamma, eps not finite and
 *   positive, context without MOE_POST_NORM).
 *
 * moe_post_norm_backward: from dout = dL/dout (bf16 [T,D], the tokens of
 *   the forward that wrote `saved`) computes, with g = gamma * dout and
 *   c[t] = mean_d g[t,d] x[t,d],
 *     dx_pre[t,d] = bf16(r[t] g[t,d] - x[t,d] r[t]^3 c[t])   (bf16 [T,D])
 *     dgamma[d]   = sum_t dout[t,d] x[t,d] r[t]               (float [D])
 *   in FP32, sums in fixed orders (bitwise reproducible).  dx_pre is the
 *   gradient to pass as `dout` to moe_backward (and to the shared expert's).
 *   dgamma is overwritten.  Enqueue only.  Errors: MOE_ERR_INVALID_ARG
 *   (null or misaligned pointer, context without MOE_TRAINING and
 *   MOE_POST_NORM, or no gamma set).
 */
MOE_API moe_status moe_ctx_set_post_norm(moe_ctx* ctx, const void* gamma, float eps);
MOE_API moe_status moe_post_norm_backward(moe_ctx* ctx, const void* saved, const void* dout, void* dx_pre,
                                          float* dgamma, cudaStream_t stream);

/* Number of kernels this context has enqueued so far (host-side count; a
 * captured call counts once at capture time). */
MOE_API uint64_t moe_ctx_launch_count(const moe_ctx* ctx);

/*
 * Upper bound on the CTAs of each persistent launch of this context (the
 * grouped GEMMs, combine, score gradient): 0, the default, is one per SM.
 * GEMMs that run on CTA pairs (clusters of two) take max_ctas / 2 clusters,
 * and at least one.  The pages have no counterpart; a caller can leave SMs
 * to work on other streams, and a test can make each CTA walk many tiles of
 * a small problem.  Results do not depend on it: every output tile is
 * computed by one CTA (or CTA pair) with the same instruction sequence.
 * Applies to calls enqueued after it (a captured graph keeps the grids it
 * was captured with).
 * Errors: MOE_ERR_INVALID_ARG for a null context or max_ctas < 0.
 */
MOE_API moe_status moe_ctx_set_max_ctas(moe_ctx* ctx, int max_ctas);

/*
 * Allocation-free inference forward.  The pages have no counterpart: this
 * entry point exists for callers that cannot allocate device memory when
 * they need the layer -- an inference engine that gives all free HBM to its
 * KV cache at start-up, a plugin handed a stream but no allocator, or a
 * latency-critical loop that must not call cudaMalloc because it can
 * synchronise the whole device.  It runs the same kernels as an inference
 * moe_forward (no saved state), in the same launch configuration, so its
 * output equals moe_forward's bit for bit; it needs no context: every
 * intermediate lives in one file-scope device array of
 * MOE_STATIC_SCRATCH_BYTES, which every GPU that loads this library holds
 * until the process exits.  It calls no cudaMalloc/cudaFree and no
 * allocating library routine.
 *   cfg         host struct: d_model, d_ff, num_experts, top_k, precision
 *               (max_tokens and MOE_TRAINING are ignored; MOE_DEBUG_CHECKS
 *               is honoured; MOE_POST_NORM, whose gamma lives in a context,
 *               returns MOE_ERR_UNSUPPORTED)
 *   T, x, topk_ids, topk_scores, W13, W2, out, call_flags: as moe_forward
 *               (W13/W2 prepared 32x32 or 1x32 for MXFP8)
 *   device_error_word  required: a 4-byte aligned device uint32 owned by
 *               the caller that receives the MOE_DEV_ERR_* bits of the call
 *               (ORed in, never cleared here: the caller reads and clears
 *               it).  NULL returns MOE_ERR_INVALID_ARG.
 * Returns MOE_ERR_CAPACITY when the call's buffers do not fit the array.
 * They need about R*(D + F + 2D) bytes for MXFP8 (R*(2D + 2F + 2D) for BF16),
 * with R = T*top_k + 31*min(num_experts, T*top_k) rounded up to 128, plus
 * 128, plus routing arrays of a few bytes per route: a decode step of up to
 * 8 tokens fits at D = 7168, F = 2048, E = 384, top_k = 6 in MXFP8.
 * The first call on a device takes the array's device address
 * (cudaGetSymbolAddress) and sets kernel attributes, so make it before any
 * stream capture.  Every call shares the array and finds the previous call's
 * contents there: calls that may overlap on the GPU race and must be
 * ordered (one stream, or events) by the caller.
 */
#define MOE_STATIC_SCRATCH_BYTES (64ull << 20)
MOE_API moe_status moe_forward_static_scratch(const moe_config* cfg, int32_t T, const void* x,
                                              const int32_t* topk_ids, const float* topk_scores,
                                              const moe_weight* W13, const moe_weight* W2, void* out,
                                              uint32_t call_flags, uint32_t* device_error_word,
                                              cudaStream_t stream);

/*
 * Activation slots: several layers' saved states packed into one buffer,
 * with save-or-replay decisions ("Dist-MoE: Speed-of-light distributed
 * Mixture-of-Experts kernels", section 04 "Activation Packing and Dynamic
 * Recompute").  The caller allocates one device buffer of `capacity` bytes
 * (base 16-byte aligned, as every saved state; offsets are multiples of 128);
 * each training forward of a stack takes its saved state at
 * base + offset from moe_slot_push, and the backwards, in reverse order,
 * give the offsets back with moe_slot_pop.
 *
 * Decision for a layer with `remaining_layers` layers still to come after
 * it in the slot, each of which needs `input_bytes` at least:
 *   full  = full_bytes, input = input_bytes, each rounded up to 128 bytes
 *           (for a layer of this library: moe_saved_state_bytes and
 *           moe_saved_input_bytes of its configuration)
 *   cursor + full + remaining_layers * input <= capacity
 *       -> full state (forward call flags 0)
 *   else cursor + input + remaining_layers * input <= capacity
 *       -> input only (*forward_flags = MOE_SAVE_INPUT_ONLY; the backward
 *          passes MOE_REPLAY_FORWARD and rebuilds the state)
 *   else MOE_ERR_CAPACITY (the slot cannot keep every layer's input).
 * The page's planner takes the decision on the device from the routed
 * rows of the step; here the state sizes use the row capacity R_cap (the
 * saved fields' addresses enter tensor maps encoded on the host), so a
 * layer's decision depends only on its configuration and is the same on
 * every step and every graph replay.
 *
 * moe_slot_init: capacity >= 0, 1 <= max_layers <= MOE_SLOT_MAX_LAYERS.
 * moe_slot_push: errors MOE_ERR_INVALID_ARG (null pointer, negative or
 *   above 2^50 byte counts, remaining_layers outside [0,
 *   MOE_SLOT_MAX_LAYERS], a slot struct not in a state moe_slot_init and
 *   push/pop leave), MOE_ERR_CAPACITY (no room, or max_layers layers already
 *   in the slot).  An input-only layer needs a MOE_REPLAY context.
 * moe_slot_pop: `offset` must be the most recent push still in the slot
 *   (MOE_ERR_INVALID_ARG otherwise); the cursor returns to it.
 * Host-only bookkeeping: no CUDA call, no device access.
 */
#define MOE_SLOT_MAX_LAYERS 64
typedef struct {
  int64_t capacity;                      /* bytes of the slot buffer           */
  int64_t cursor;                        /* next free byte (multiple of 128)   */
  int32_t layers;                        /* saved states now in the slot       */
  int32_t max_layers;                    /* bound on `layers`                   */
  int64_t offset[MOE_SLOT_MAX_LAYERS];   /* offset of each stacked state        */
  uint32_t flags[MOE_SLOT_MAX_LAYERS];   /* its forward call flags              */
} moe_slot;

/* Bytes of an input-only saved state (routing fields, scores, the
 * pre-norm output under MOE_POST_NORM, and x) and one field's place in it. */
MOE_API size_t moe_saved_input_bytes(const moe_config* cfg);
MOE_API moe_status moe_saved_input_field(const moe_config* cfg, int field, size_t* offset, size_t* bytes);

MOE_API moe_status moe_slot_init(moe_slot* slot, int64_t capacity, int32_t max_layers);
MOE_API moe_status moe_slot_push(moe_slot* slot, int64_t full_bytes, int64_t input_bytes, int32_t remaining_layers,
                                 int64_t* offset, uint32_t* forward_flags);
MOE_API moe_status moe_slot_pop(moe_slot* slot, int64_t offset);

/* Library version string. */
MOE_API const char* moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
