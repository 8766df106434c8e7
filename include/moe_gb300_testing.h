/*
 * moe_gb300_testing.h -- inspection entry points for tests (not the product
 * interface of moe_gb300.h).
 *
 * They read the scratch regions of a context and copy device memory to the
 * host synchronously, so that parity tests can compare intermediate stages
 * (gathered bundles, scale atoms, the inference routing copy) with the
 * oracle.  No call of the hot path uses them, and none may be made inside
 * stream capture.  The library exports them next to the boundary calls.
 */
#ifndef MOE_GB300_TESTING_H
#define MOE_GB300_TESTING_H

#include "moe_gb300.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Copy `bytes` from device memory to host memory (synchronous).  A helper
 * for tests that inspect scratch; not part of the hot path. */
MOE_API moe_status moe_debug_copy_to_host(void* host_dst, const void* dev_src, size_t bytes);

/* Scratch regions of a context, for inspection by tests.  Sizes follow
 * R_cap (moe_row_capacity) and B_cap = (T_max*K + 31*E)/128 + E + 1. */
typedef enum {
  MOE_BUF_XROW = 0,        /* gathered x row bundle: bf16 [R_cap, D] or e4m3
                              (MOE_NVFP4: chunks [B_cap][D/64] of 4608 bytes)  */
  MOE_BUF_XROW_SCALE = 1,  /* e8m0 row-bundle atoms [B_cap][D/128]
                              (MOE_NVFP4: FP32 row scales [R_cap])             */
  MOE_BUF_H2ROW = 2,       /* h2 row bundle: bf16 [R_cap, F] or e4m3
                              (MOE_NVFP4: chunks [B_cap][F/64])                */
  MOE_BUF_H2ROW_SCALE = 3, /* e8m0 row-bundle atoms [B_cap][F/128]
                              (MOE_NVFP4: FP32 row scales [R_cap])             */
  MOE_BUF_H3 = 4,          /* bf16 [R_cap, D]                                  */
  MOE_BUF_DH3ROW = 5,      /* bf16 [R_cap, D] or e4m3                          */
  MOE_BUF_DH3ROW_SCALE = 6,/* e8m0 row-bundle atoms [B_cap][D/128]            */
  MOE_BUF_DH3COL = 7,      /* bf16 [D, R_cap] or e4m3                          */
  MOE_BUF_DH3COL_SCALE = 8,/* e8m0 column-bundle atoms [D/128][B_cap]         */
  MOE_BUF_DH1ROW = 9,      /* bf16 [R_cap, 2F] or e4m3                         */
  MOE_BUF_DH1ROW_SCALE = 10,/* e8m0 row-bundle atoms [B_cap][2F/128]          */
  MOE_BUF_DH1COL = 11,     /* bf16 [2F, R_cap] or e4m3                         */
  MOE_BUF_DH1COL_SCALE = 12,/* e8m0 column-bundle atoms [2F/128][B_cap]       */
  MOE_BUF_DXR = 13,        /* bf16 [R_cap, D]                                  */
  MOE_BUF_ROUTING = 14,    /* inference routing state (same layout as saved)   */
  MOE_BUF_ERROR = 15,      /* uint32 error word                                */
  MOE_BUF_NORM = 16,       /* MOE_POST_NORM training: float r[T_max], then the
                              dgamma partial sums [ceil(T_max/64)][D]          */
  MOE_BUF_REPLAY = 17,     /* MOE_REPLAY: a full saved state (same layout) that
                              a backward with MOE_REPLAY_FORWARD rebuilds       */
  MOE_BUF_SYNC = 18,       /* int32 counters of the single-launch forward:
                              3 + 2*B_cap words, zero between launches          */
  MOE_BUF_H2F = 19,        /* MOE_NVFP4: FP32 h2 [R_cap, F] (then quantised)   */
  MOE_BUF_NUM = 20
} moe_buffer;

MOE_API moe_status moe_ctx_buffer(moe_ctx* ctx, int which, void** dev_ptr, size_t* bytes);

/* Failure test of the single-launch forward (MOE_FUSED_LAUNCH): with
 * stall != 0 its W2 tiles wait for one more finished W13 tile than exists
 * (a count nothing reaches), so their waits run out; every counter wait of
 * that launch gives up after wait_cycles SM cycles (> 0; the default is
 * about 2 s) and sets MOE_DEV_ERR_TIMEOUT.  stall = 0 and wait_cycles = 0
 * restore the defaults.  Applies to later calls; no device access. */
MOE_API moe_status moe_ctx_test_fused_stall(moe_ctx* ctx, int stall, int64_t wait_cycles);

/* Tiles of the grouped GEMMs whose weight is the A operand (forward W13 and
 * W2, W13 input gradient): mode 1 takes one routing row block (<= 128 rows)
 * as the B operand; mode 2 takes row-block pairs (two consecutive blocks of
 * one expert, <= 256 rows, the pairs of MOE_SAVED_BLOCKS word 3); mode 3
 * runs the forward's pairs on CTA pairs (clusters of two CTAs, one 256 x 256
 * tensor-core instruction over both: each CTA one A tile and one block of
 * the pair; a GEMM whose K is not a multiple of 256 bytes, or W2 where
 * d_model is not a multiple of 256, takes mode 2's tiles; the backward as
 * mode 2); mode 0 (the default) takes CTA pairs for the forward when
 * max_tokens * top_k >= 192 * num_experts in MXFP8 or >= 128 * num_experts
 * in BF16, and in BF16 pairs for the backward from the same density.
 * All give the same results bit for bit, and a forward and its backward
 * may run in different modes (both read the same saved state).  Applies to
 * later calls; no device access. */
MOE_API moe_status moe_ctx_test_tile_mode(moe_ctx* ctx, int mode);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_TESTING_H */
