// C ABI of the MoE layer: context (fixed scratch), saved-state layout,
// weight preparation, and the forward/backward launch sequences.
//
// Forward (one stream, no host synchronisation):
//   route -> gather x (row bundle; + column bundle when training)
//   -> W13 GEMM with fused SwiGLU -> W2 GEMM -> combine.
// Backward:
//   [replay: gather x -> W13 GEMM (-> W2 GEMM) into the context's replay
//   scratch, for a forward that saved only its input]
//   dh3 gather (row + column bundles) -> W2 DGRAD with fused SwiGLU backward
//   -> W2 WGRAD -> W13 DGRAD -> W13 WGRAD -> K-reduction of dX.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "kernels.cuh"
#include "moe_gb300.h"
#include "moe_gb300_testing.h"

using namespace moe;

struct moe_ctx {
  moe_config cfg;
  int device;
  int num_sms;
  int max_ctas = 0;   // moe_ctx_set_max_ctas (0: num_sms)
  int fused_stall = 0;             // moe_ctx_test_fused_stall
  // grouped-M GEMM tiles over row-block pairs (B up to 256 rows): chosen at
  // creation for BF16 when the capacity gives the experts 128 routes each on
  // average (max_tokens * top_k >= 128 E); moe_ctx_test_tile_mode overrides it
  bool pair_tiles_auto = false;
  // the forward's GEMMs over row-block pairs on CTA pairs, chosen at creation
  // when the capacity gives the experts 192 (MXFP8) or 128 (BF16) routes on
  // average; moe_ctx_test_tile_mode overrides it
  bool cta_pairs_auto = false;
  int tile_mode = 0;               // 0: automatic, 1: row blocks, 2: pairs, 3: pairs on CTA pairs
  long long fused_wait = 0;        // counter-wait limit of the single-launch forward (0: default)
  const void* norm_gamma = nullptr;   // moe_ctx_set_post_norm (MOE_POST_NORM)
  float norm_eps = 0.0f;
  int64_t r_cap;
  int64_t b_cap;
  uint8_t* base;
  size_t bytes;
  void* buf[MOE_BUF_NUM];
  size_t buf_bytes[MOE_BUF_NUM];
  uint32_t* err;
  unsigned long long* clip;   // [2] clamped gate / up counts (clip statistics)
  bool timing;          // calls record the stage events
  bool events;          // the stage events exist (created once, destroyed with the context)
  cudaEvent_t ev[2][8];
  uint64_t launches;
  // saved-state pointer -> written input-only (MOE_SAVE_INPUT_ONLY) by the
  // last forward of this context that wrote there
  std::unordered_map<const void*, bool> saved_input_only;
};

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool config_ok(const moe_config* c) {
  if (!c) return false;
  if (c->max_tokens < 1 || c->top_k < 1 || c->top_k > 32) return false;
  if (c->num_experts < 1 || c->num_experts > 1024) return false;
  if (c->d_model < 128 || c->d_ff < 128) return false;
  if (c->precision != MOE_BF16 && c->precision != MOE_MXFP8 && c->precision != MOE_NVFP4) return false;
  if (!(c->swiglu_limit >= 0.0f) || c->swiglu_limit > 3.0e38f) return false;   // also rejects NaN
  const int64_t routes = static_cast<int64_t>(c->max_tokens) * c->top_k;
  if (routes + 31LL * c->num_experts > (1LL << 28)) return false;
  return true;
}

bool config_tileable(const moe_config* c) { return c->d_model % 128 == 0 && c->d_ff % 128 == 0; }

bool use_pairs(const moe_ctx* c) { return c->tile_mode >= 2 || (c->tile_mode == 0 && c->pair_tiles_auto); }

// Tiles of the forward's grouped-M GEMMs (W13 + SwiGLU, W2): row blocks, row-
// block pairs, or row-block pairs on CTA pairs.
GemmMode forward_tiles(const moe_ctx* c) {
  switch (c->tile_mode) {
    case 1: return kGroupedM;
    case 2: return kGroupedMP;
    case 3: return kGroupedMC;
    default:
      if (c->cta_pairs_auto) return kGroupedMC;
      return c->pair_tiles_auto ? kGroupedMP : kGroupedM;
  }
}

int64_t row_cap(const moe_config* c) {
  const int64_t r = static_cast<int64_t>(c->max_tokens) * c->top_k + 31LL * c->num_experts;
  return static_cast<int64_t>(align_up(static_cast<size_t>(r), 128)) + 128;  // +128: slack for the last stage
}

int64_t block_cap(const moe_config* c) {
  const int64_t r = static_cast<int64_t>(c->max_tokens) * c->top_k + 31LL * c->num_experts;
  return r / 128 + c->num_experts + 1;
}

struct SavedLayout {
  size_t off[MOE_SAVED_NUM_FIELDS];
  size_t size[MOE_SAVED_NUM_FIELDS];
  size_t routing_bytes;  // header .. scores
  size_t total;
};

// The full state (input_only false) or the input-only state a forward with
// MOE_SAVE_INPUT_ONLY writes: the same routing fields and PRENORM at the
// same offsets, then the expert state or the copy of x.
SavedLayout saved_layout(const moe_config* c, bool input_only = false) {
  SavedLayout L{};
  const int64_t R = row_cap(c), B = block_cap(c);
  const int64_t E = c->num_experts, TK = static_cast<int64_t>(c->max_tokens) * c->top_k;
  const int64_t D = c->d_model, F = c->d_ff;
  const bool mx = c->precision == MOE_MXFP8;
  const size_t esz = mx ? 1 : 2;
  size_t sz[MOE_SAVED_NUM_FIELDS] = {};
  sz[MOE_SAVED_HEADER] = 16 * sizeof(int);
  sz[MOE_SAVED_COUNTS] = E * sizeof(int);
  sz[MOE_SAVED_OFFSETS] = (E + 1) * sizeof(int);
  sz[MOE_SAVED_POFFSETS] = (E + 1) * sizeof(int);
  sz[MOE_SAVED_PERM] = R * sizeof(int);
  sz[MOE_SAVED_INV] = TK * sizeof(int);
  sz[MOE_SAVED_BLOCKS] = B * 4 * sizeof(int);
  sz[MOE_SAVED_SCORES] = TK * sizeof(float);
  sz[MOE_SAVED_BSTART] = (E + 1) * sizeof(int);
  sz[MOE_SAVED_ROWBLOCK] = (R / 32) * sizeof(int);
  sz[MOE_SAVED_H1] = R * 2 * F * 2;
  sz[MOE_SAVED_XCOL] = D * R * esz;
  sz[MOE_SAVED_XCOL_SCALE] = mx ? (D / 128) * B * 512 : 0;
  sz[MOE_SAVED_H2COL] = F * R * esz;
  sz[MOE_SAVED_H2COL_SCALE] = mx ? (F / 128) * B * 512 : 0;
  sz[MOE_SAVED_H3] = R * D * 2;
  sz[MOE_SAVED_PRENORM] = (c->flags & MOE_POST_NORM) ? static_cast<int64_t>(c->max_tokens) * D * 2 : 0;
  if (input_only) {
    for (int f : {MOE_SAVED_H1, MOE_SAVED_XCOL, MOE_SAVED_XCOL_SCALE, MOE_SAVED_H2COL, MOE_SAVED_H2COL_SCALE,
                  MOE_SAVED_H3})
      sz[f] = 0;
    sz[MOE_SAVED_X] = static_cast<int64_t>(c->max_tokens) * D * 2;
  }
  // routing fields first (the inference copy in the context holds just these)
  static const int order[MOE_SAVED_NUM_FIELDS] = {
      MOE_SAVED_HEADER,   MOE_SAVED_COUNTS, MOE_SAVED_OFFSETS, MOE_SAVED_POFFSETS,   MOE_SAVED_PERM,
      MOE_SAVED_INV,      MOE_SAVED_BLOCKS, MOE_SAVED_SCORES,  MOE_SAVED_BSTART,     MOE_SAVED_ROWBLOCK,
      MOE_SAVED_PRENORM,  MOE_SAVED_H1,     MOE_SAVED_XCOL,    MOE_SAVED_XCOL_SCALE, MOE_SAVED_H2COL,
      MOE_SAVED_H2COL_SCALE, MOE_SAVED_H3,  MOE_SAVED_X};
  size_t off = 0;
  for (int k = 0; k < MOE_SAVED_NUM_FIELDS; ++k) {
    const int i = order[k];
    L.off[i] = off;
    L.size[i] = sz[i];
    off += align_up(sz[i], kAlign);
    if (i == MOE_SAVED_ROWBLOCK) L.routing_bytes = off;
  }
  L.total = off;
  return L;
}

struct ScratchLayout {
  size_t off[MOE_BUF_NUM];
  size_t size[MOE_BUF_NUM];
  size_t total;
};

ScratchLayout scratch_layout(const moe_config* c) {
  ScratchLayout L{};
  const int64_t R = row_cap(c), B = block_cap(c);
  const int64_t D = c->d_model, F = c->d_ff;
  const bool mx = c->precision == MOE_MXFP8;
  const bool train = (c->flags & MOE_TRAINING) != 0;
  const size_t esz = mx ? 1 : 2;
  size_t sz[MOE_BUF_NUM] = {};
  sz[MOE_BUF_XROW] = R * D * esz;
  sz[MOE_BUF_XROW_SCALE] = mx ? B * (D / 128) * 512 : 0;
  sz[MOE_BUF_H2ROW] = R * F * esz;
  sz[MOE_BUF_H2ROW_SCALE] = mx ? B * (F / 128) * 512 : 0;
  sz[MOE_BUF_H3] = R * D * 2;
  if (train) {
    sz[MOE_BUF_DH3ROW] = R * D * esz;
    sz[MOE_BUF_DH3ROW_SCALE] = mx ? B * (D / 128) * 512 : 0;
    sz[MOE_BUF_DH3COL] = D * R * esz;
    sz[MOE_BUF_DH3COL_SCALE] = mx ? (D / 128) * B * 512 : 0;
    sz[MOE_BUF_DH1ROW] = R * 2 * F * esz;
    sz[MOE_BUF_DH1ROW_SCALE] = mx ? B * (2 * F / 128) * 512 : 0;
    sz[MOE_BUF_DH1COL] = 2 * F * R * esz;
    sz[MOE_BUF_DH1COL_SCALE] = mx ? (2 * F / 128) * B * 512 : 0;
    sz[MOE_BUF_DXR] = R * D * 2;
  }
  if (train && (c->flags & MOE_POST_NORM)) {   // r[T_max], then the dgamma slab partials
    const int64_t Tm = c->max_tokens;
    sz[MOE_BUF_NORM] = (Tm + (Tm + kPostNormSlab - 1) / kPostNormSlab * D) * sizeof(float);
  }
  if (train && (c->flags & MOE_REPLAY)) sz[MOE_BUF_REPLAY] = saved_layout(c).total;
  sz[MOE_BUF_ROUTING] = saved_layout(c).routing_bytes;
  if (!train && mx) sz[MOE_BUF_SYNC] = (3 + 2 * B) * sizeof(int);   // single-launch forward counters
  sz[MOE_BUF_ERROR] = 32;   // error word at 0, clip counters at 16
  if (c->precision == MOE_NVFP4) {
    // inference only: chunks of the routing blocks' x and h2 rows with their
    // FP32 row scales, and the FP32 h2 the W13 epilogue writes
    sz[MOE_BUF_XROW] = nvfp4_chunk_bytes(B, static_cast<int>(D));
    sz[MOE_BUF_XROW_SCALE] = R * sizeof(float);
    sz[MOE_BUF_H2ROW] = nvfp4_chunk_bytes(B, static_cast<int>(F));
    sz[MOE_BUF_H2ROW_SCALE] = R * sizeof(float);
    sz[MOE_BUF_H2F] = R * F * sizeof(float);
  }
  size_t off = 0;
  for (int i = 0; i < MOE_BUF_NUM; ++i) {
    L.off[i] = off;
    L.size[i] = sz[i];
    off += align_up(sz[i], kAlign);
  }
  L.total = off;
  return L;
}

RoutingPtrs routing_ptrs(uint8_t* base, const SavedLayout& L) {
  RoutingPtrs r;
  r.hdr = reinterpret_cast<int*>(base + L.off[MOE_SAVED_HEADER]);
  r.counts = reinterpret_cast<int*>(base + L.off[MOE_SAVED_COUNTS]);
  r.offsets = reinterpret_cast<int*>(base + L.off[MOE_SAVED_OFFSETS]);
  r.poffsets = reinterpret_cast<int*>(base + L.off[MOE_SAVED_POFFSETS]);
  r.perm = reinterpret_cast<int*>(base + L.off[MOE_SAVED_PERM]);
  r.inv = reinterpret_cast<int*>(base + L.off[MOE_SAVED_INV]);
  r.blocks = reinterpret_cast<int4*>(base + L.off[MOE_SAVED_BLOCKS]);
  r.scores = reinterpret_cast<float*>(base + L.off[MOE_SAVED_SCORES]);
  r.bstart = reinterpret_cast<int*>(base + L.off[MOE_SAVED_BSTART]);
  r.row_block = reinterpret_cast<int*>(base + L.off[MOE_SAVED_ROWBLOCK]);
  return r;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(x)                          \
  do {                                      \
    const cudaError_t _e = (x);             \
    if (_e != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

#define MOE_PASS(x)                         \
  do {                                      \
    const moe_status _s = (x);              \
    if (_s != MOE_OK) return _s;            \
  } while (0)

// need_t: the backward's transposed copy is needed (which a 1x32 inference
// weight does not have); an MXFP8 context's forward also takes 1x32 weights.
bool weight_ok(const moe_weight* w, moe_precision prec, int E, int N, int K, bool need_t) {
  if (!w || w->E != E || w->N != N || w->K != K) return false;
  const bool row32 = prec == MOE_MXFP8 && !need_t && w->precision == MOE_MXFP8_1X32;
  if (w->precision != prec && !row32) return false;
  if (!w->data || !aligned16(w->data)) return false;
  if ((prec == MOE_MXFP8 || prec == MOE_NVFP4) && (!w->scale || !aligned16(w->scale))) return false;
  if (need_t) {
    // MXFP8: the input-gradient scale atoms, and either the transposed codes
    // (a K-major input-gradient operand) or none (the GEMM reads the
    // forward's codes MN-major); BF16: the transposed copy
    if (prec == MOE_MXFP8) {
      if (!w->scale_t || !aligned16(w->scale_t) || (w->data_t && !aligned16(w->data_t))) return false;
    } else if (!w->data_t || !aligned16(w->data_t)) {
      return false;
    }
  }
  return true;
}

uint8_t* B(moe_ctx* c, int which) { return static_cast<uint8_t*>(c->buf[which]); }

// Record stage event `idx` of `pass` (0 forward, 1 backward) when timing is on.
cudaError_t stage_mark(moe_ctx* c, int pass, int idx, cudaStream_t s) {
  if (!c->timing) return cudaSuccess;
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &st);
  if (e != cudaSuccess) return e;
  if (st == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(c->ev[pass][idx], s, cudaEventRecordExternal);
  return cudaEventRecord(c->ev[pass][idx], s);
}

// The W13 + SwiGLU GEMM of a forward (or replay) into *g1: x row bundle
// from scratch, h2 row bundle to scratch; with `act` (a full saved state),
// also h1 and the h2 column bundle into act's fields.  False if a tensor map
// cannot be encoded.
bool fill_w13(moe_ctx* ctx, const RoutingPtrs& rp, const moe_weight* W13, uint8_t* act, const SavedLayout& SL,
              bool marks, GemmLaunch* g1, GemmMode mode) {
  const moe_config& c = ctx->cfg;
  const int D = c.d_model, F = c.d_ff, E = c.num_experts;
  const bool mx = c.precision == MOE_MXFP8;
  const int64_t R = ctx->r_cap;
  if (mode == kGroupedMC && D % (mx ? 256 : 128) != 0) mode = kGroupedMP;   // a CTA pair's stage: 256 bytes of K
  g1->mx = mx;
  g1->na = mode == kGroupedM ? 2 : 1;
  g1->epi = kEpiSwigluFwd;
  g1->mode = mode;
  if (!make_tmap(&g1->tmA, W13->data, mx, static_cast<int64_t>(E) * 2 * F, D, 128) ||
      !make_tmap(&g1->tmB, B(ctx, MOE_BUF_XROW), mx, R, D, 32) ||
      !make_grouped_m_boxes(g1, W13->data, static_cast<int64_t>(E) * 2 * F, W13->scale, B(ctx, MOE_BUF_XROW), R,
                            mx, D, F))
    return false;
  GemmParams& p1 = g1->p;
  p1.hdr = rp.hdr;
  p1.blocks = rp.blocks;
  p1.poffsets = rp.poffsets;
  p1.E = E;
  p1.b_box_rows = 32;
  p1.n_tiles = F / (mode == kGroupedMP ? 64 : 128);   // (CTA pairs: 2 x 64 features)
  p1.K = D;
  p1.a_rows_per_expert = 2 * F;
  p1.a_up_offset = F;
  p1.sfa = W13->scale;
  p1.sfa_ts = D / 128;
  p1.sfb = B(ctx, MOE_BUF_XROW_SCALE);
  p1.sfb_ts = D / 128;
  p1.out0 = B(ctx, MOE_BUF_H2ROW);
  p1.out0_pitch = F;
  p1.out0_sf = B(ctx, MOE_BUF_H2ROW_SCALE);
  p1.out0_sf_kg = F / 128;
  p1.b_cap = static_cast<int>(ctx->b_cap);
  if (act) {
    p1.out1 = act + SL.off[MOE_SAVED_H2COL];
    p1.out1_pitch = R;
    p1.out1_sf = mx ? act + SL.off[MOE_SAVED_H2COL_SCALE] : nullptr;
    p1.h1 = reinterpret_cast<__nv_bfloat16*>(act + SL.off[MOE_SAVED_H1]);
    p1.h1_pitch = 2 * F;
  }
  p1.F = F;
  p1.save_h1 = act ? 1 : 0;
  p1.want_col = act ? 1 : 0;
  p1.swiglu_limit = c.swiglu_limit;
  p1.clip = (marks && c.swiglu_limit > 0.0f) ? ctx->clip : nullptr;   // a replay counts no clips again
  p1.err = ctx->err;
  g1->max_tiles = static_cast<int>(ctx->b_cap * p1.n_tiles);
  return true;
}

// The W2 GEMM into *g2: h3 = h2 W2[e]^T from the h2 row bundle in scratch.
bool fill_w2(moe_ctx* ctx, const RoutingPtrs& rp, const moe_weight* W2, uint8_t* h3, GemmLaunch* g2,
             GemmMode mode) {
  const moe_config& c = ctx->cfg;
  const int D = c.d_model, F = c.d_ff, E = c.num_experts;
  const bool mx = c.precision == MOE_MXFP8;
  const int64_t R = ctx->r_cap;
  // a CTA pair's tile is 256 features, its stage 256 bytes of K
  if (mode == kGroupedMC && (D % 256 != 0 || F % (mx ? 256 : 128) != 0)) mode = kGroupedMP;
  g2->mx = mx;
  g2->na = mode == kGroupedM ? pair_tiles(D) : 1;
  g2->epi = kEpiStore;
  g2->mode = mode;
  if (!make_tmap(&g2->tmA, W2->data, mx, static_cast<int64_t>(E) * D, F, 128) ||
      !make_tmap(&g2->tmB, B(ctx, MOE_BUF_H2ROW), mx, R, F, 32) ||
      !make_grouped_m_boxes(g2, W2->data, static_cast<int64_t>(E) * D, W2->scale, B(ctx, MOE_BUF_H2ROW), R, mx, F))
    return false;
  GemmParams& p2 = g2->p;
  p2.hdr = rp.hdr;
  p2.blocks = rp.blocks;
  p2.poffsets = rp.poffsets;
  p2.E = E;
  p2.b_box_rows = 32;
  p2.n_tiles = D / (mode == kGroupedMC ? 256 : 128 * g2->na);   // (CTA pairs: 2 x 128 features)
  p2.K = F;
  p2.a_rows_per_expert = D;
  p2.sfa = W2->scale;
  p2.sfa_ts = F / 128;
  p2.sfb = B(ctx, MOE_BUF_H2ROW_SCALE);
  p2.sfb_ts = F / 128;
  p2.out0 = h3;
  p2.out0_pitch = D;
  p2.F = F;
  p2.err = ctx->err;
  g2->max_tiles = static_cast<int>(ctx->b_cap * p2.n_tiles);
  return true;
}

// Gather x (the row bundle; with `act`, also the column bundle into act's
// XCOL fields) and run the W13 + SwiGLU GEMM (with `act`, h1 and the h2
// column bundle into act's fields).  `act` is a full saved state (a
// training forward's, or the context's replay scratch) or null (inference,
// input-only states).  `marks`: record the forward's stage events and count
// clip statistics (off when a backward replays these stages).
moe_status run_gather_w13(moe_ctx* ctx, const void* x, const RoutingPtrs& rp, const moe_weight* W13, uint8_t* act,
                          const SavedLayout& SL, bool marks, int sms, cudaStream_t stream) {
  const moe_config& c = ctx->cfg;
  const int D = c.d_model, K = c.top_k;
  const bool mx = c.precision == MOE_MXFP8;
  const int64_t R = ctx->r_cap;
  if (act) {
    // row bundle (W13 operand) and column bundle (W13 WGRAD operand) in one pass
    CUtensorMap tr, tc;
    if (mx && (!make_tmap(&tr, B(ctx, MOE_BUF_XROW), true, R, D, 128) ||
               !make_tmap(&tc, act + SL.off[MOE_SAVED_XCOL], true, D, R, 128)))
      return MOE_ERR_CUDA;
    MOE_TRY(launch_gather_both(mx, false, x, D, K, rp, B(ctx, MOE_BUF_XROW), B(ctx, MOE_BUF_XROW_SCALE),
                               act + SL.off[MOE_SAVED_XCOL], mx ? act + SL.off[MOE_SAVED_XCOL_SCALE] : nullptr,
                               static_cast<int>(R), static_cast<int>(ctx->b_cap), sms, stream, &tr, &tc));
  } else {
    MOE_TRY(launch_gather_rows(mx, false, x, D, K, rp, B(ctx, MOE_BUF_XROW), B(ctx, MOE_BUF_XROW_SCALE),
                               static_cast<int>(R), sms, stream));
  }
  ctx->launches += 1;
  if (marks) MOE_TRY(stage_mark(ctx, 0, 2, stream));

  // ---- W13 + SwiGLU
  GemmLaunch g1{};
  if (!fill_w13(ctx, rp, W13, act, SL, marks, &g1, forward_tiles(ctx))) return MOE_ERR_CUDA;
  MOE_TRY(launch_gemm(g1, sms, stream));
  ctx->launches += 1;
  if (marks) MOE_TRY(stage_mark(ctx, 0, 3, stream));
  return MOE_OK;
}

// The W2 GEMM: h3 = h2 W2[e]^T from the h2 row bundle in scratch.
moe_status run_w2(moe_ctx* ctx, const RoutingPtrs& rp, const moe_weight* W2, uint8_t* h3, int sms,
                  cudaStream_t stream) {
  GemmLaunch g2{};
  if (!fill_w2(ctx, rp, W2, h3, &g2, forward_tiles(ctx))) return MOE_ERR_CUDA;
  MOE_TRY(launch_gemm(g2, sms, stream));
  ctx->launches += 1;
  return MOE_OK;
}
// NVFP4 inference after routing (nvfp4.cu): the routed x rows quantised
// into their routing blocks' chunks; the W13 + SwiGLU GEMM to FP32 h2 and
// the h2 rows quantised (one stage); the W2 GEMM to BF16 h3.  Grids: one CTA
// per SM at most, and no more than the tiles the token count allows.
moe_status run_nvfp4(moe_ctx* ctx, int T, const void* x, const RoutingPtrs& rp, const moe_weight* W13,
                     const moe_weight* W2, int sms, cudaStream_t stream) {
  const moe_config& c = ctx->cfg;
  const int D = c.d_model, F = c.d_ff, K = c.top_k;
  const int R = static_cast<int>(ctx->r_cap);
  float* gx = reinterpret_cast<float*>(B(ctx, MOE_BUF_XROW_SCALE));
  float* gh = reinterpret_cast<float*>(B(ctx, MOE_BUF_H2ROW_SCALE));
  MOE_TRY(launch_nvfp4_rows(false, x, D, K, rp, R, B(ctx, MOE_BUF_XROW), gx, sms, stream));
  ctx->launches += 1;
  MOE_TRY(stage_mark(ctx, 0, 2, stream));
  const int64_t tk = static_cast<int64_t>(T) * K;
  const int64_t max_blocks = tk / 128 + std::min<int64_t>(c.num_experts, tk) + 1;
  Fp4GemmParams p{};
  p.a = static_cast<const uint8_t*>(W13->data);
  p.ga = reinterpret_cast<const float*>(W13->scale);
  p.b = B(ctx, MOE_BUF_XROW);
  p.gb = gx;
  p.hdr = rp.hdr;
  p.blocks = rp.blocks;
  p.out = B(ctx, MOE_BUF_H2F);
  p.ks = D / 64;
  p.n_tiles = F / 128;
  p.a_tiles_e = 2 * F / 128;
  p.ld = F;
  p.swiglu_limit = c.swiglu_limit;
  p.clip = ctx->clip;
  p.err = ctx->err;
  MOE_TRY(launch_nvfp4_gemm(p, true, static_cast<int>(std::min<int64_t>(sms, max_blocks * p.n_tiles)), stream));
  MOE_TRY(launch_nvfp4_rows(true, B(ctx, MOE_BUF_H2F), F, K, rp, R, B(ctx, MOE_BUF_H2ROW), gh, sms, stream));
  ctx->launches += 2;
  MOE_TRY(stage_mark(ctx, 0, 3, stream));
  p.a = static_cast<const uint8_t*>(W2->data);
  p.ga = reinterpret_cast<const float*>(W2->scale);
  p.b = B(ctx, MOE_BUF_H2ROW);
  p.gb = gh;
  p.out = B(ctx, MOE_BUF_H3);
  p.ks = F / 64;
  p.n_tiles = D / 128;
  p.a_tiles_e = D / 128;
  p.ld = D;
  p.clip = nullptr;
  MOE_TRY(launch_nvfp4_gemm(p, false, static_cast<int>(std::min<int64_t>(sms, max_blocks * p.n_tiles)), stream));
  ctx->launches += 1;
  return MOE_OK;
}

// The whole inference forward as one launch (MOE_FUSED_LAUNCH): the same
// tensor maps and GEMM parameters as the staged launches, and the counters
// in the context's sync buffer.
moe_status run_fused_forward(moe_ctx* ctx, int T, const void* x, const int32_t* ids, const float* scores,
                             const RoutingPtrs& rp, const moe_weight* W13, const moe_weight* W2, void* out,
                             bool accumulate, int sms, cudaStream_t stream) {
  const moe_config& c = ctx->cfg;
  const SavedLayout SL = saved_layout(&c);
  GemmLaunch g1{}, g2{};
  if (!fill_w13(ctx, rp, W13, nullptr, SL, true, &g1, kGroupedM) ||
      !fill_w2(ctx, rp, W2, B(ctx, MOE_BUF_H3), &g2, kGroupedM))
    return MOE_ERR_CUDA;
  if (g1.p.a_pair_box != 2 || g2.p.a_pair_box != 1 || !g1.p.b_full_box || !g2.p.b_full_box)
    return MOE_ERR_UNSUPPORTED;
  FusedLaunch L{};
  L.a13 = g1.aux[0];
  L.sf13 = g1.aux[2];
  L.bx32 = g1.tmB;
  L.bx128 = g1.aux[1];
  L.a2 = g2.aux[0];
  L.sf2 = g2.aux[2];
  L.bh32 = g2.tmB;
  L.bh128 = g2.aux[1];
  FusedArgs& a = L.args;
  a.ids = ids;
  a.scores = scores;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.T = T;
  a.K = c.top_k;
  a.E = c.num_experts;
  a.D = c.d_model;
  a.F = c.d_ff;
  a.debug = (c.flags & MOE_DEBUG_CHECKS) ? 1 : 0;
  a.accumulate = accumulate ? 1 : 0;
  a.rp = rp;
  a.xrow = B(ctx, MOE_BUF_XROW);
  a.xsf = B(ctx, MOE_BUF_XROW_SCALE);
  a.sync = reinterpret_cast<int*>(B(ctx, MOE_BUF_SYNC));
  a.b_cap = static_cast<int>(ctx->b_cap);
  a.wait_cycles = ctx->fused_wait > 0 ? ctx->fused_wait : kWaitTimeoutCycles;
  a.stall = ctx->fused_stall;
  a.g13 = g1.p;
  a.g2 = g2.p;
  const int64_t tk = static_cast<int64_t>(T) * c.top_k;
  L.max_blocks = static_cast<int>(tk / 128 + std::min<int64_t>(c.num_experts, tk) + 1);
  MOE_TRY(launch_fused_forward(L, sms, stream));
  ctx->launches += 1;
  return MOE_OK;
}

}  // namespace

// =================================================================== ABI

extern "C" {

const char* moe_version(void) { return "moe_gb300 0.1 (sm_103a)"; }

int64_t moe_row_capacity(const moe_config* cfg) { return config_ok(cfg) ? row_cap(cfg) : 0; }

size_t moe_saved_state_bytes(const moe_config* cfg) { return config_ok(cfg) ? saved_layout(cfg).total : 0; }

moe_status moe_saved_state_field(const moe_config* cfg, int field, size_t* offset, size_t* bytes) {
  if (!config_ok(cfg) || field < 0 || field >= MOE_SAVED_NUM_FIELDS || !offset || !bytes)
    return MOE_ERR_INVALID_ARG;
  const SavedLayout L = saved_layout(cfg);
  *offset = L.off[field];
  *bytes = L.size[field];
  return MOE_OK;
}

size_t moe_saved_input_bytes(const moe_config* cfg) { return config_ok(cfg) ? saved_layout(cfg, true).total : 0; }

moe_status moe_saved_input_field(const moe_config* cfg, int field, size_t* offset, size_t* bytes) {
  if (!config_ok(cfg) || field < 0 || field >= MOE_SAVED_NUM_FIELDS || !offset || !bytes)
    return MOE_ERR_INVALID_ARG;
  const SavedLayout L = saved_layout(cfg, true);
  *offset = L.off[field];
  *bytes = L.size[field];
  return MOE_OK;
}

// ---- activation slots: host bookkeeping of the save-or-replay decisions

moe_status moe_slot_init(moe_slot* slot, int64_t capacity, int32_t max_layers) {
  if (!slot || capacity < 0 || max_layers < 1 || max_layers > MOE_SLOT_MAX_LAYERS) return MOE_ERR_INVALID_ARG;
  std::memset(slot, 0, sizeof(*slot));
  slot->capacity = capacity;
  slot->max_layers = max_layers;
  return MOE_OK;
}

moe_status moe_slot_push(moe_slot* slot, int64_t full_bytes, int64_t input_bytes, int32_t remaining_layers,
                         int64_t* offset, uint32_t* forward_flags) {
  if (!slot || !offset || !forward_flags || full_bytes < 0 || input_bytes < 0 || remaining_layers < 0)
    return MOE_ERR_INVALID_ARG;
  if (full_bytes > (int64_t{1} << 50) || input_bytes > (int64_t{1} << 50) || remaining_layers > MOE_SLOT_MAX_LAYERS)
    return MOE_ERR_INVALID_ARG;   // keeps the sums below far from overflow
  if (slot->layers < 0 || slot->max_layers < 1 || slot->max_layers > MOE_SLOT_MAX_LAYERS ||
      slot->layers > slot->max_layers || slot->cursor < 0 || slot->cursor > slot->capacity)
    return MOE_ERR_INVALID_ARG;
  if (slot->layers == slot->max_layers) return MOE_ERR_CAPACITY;
  const int64_t full = static_cast<int64_t>(align_up(static_cast<size_t>(full_bytes), 128));
  const int64_t input = static_cast<int64_t>(align_up(static_cast<size_t>(input_bytes), 128));
  const int64_t reserve = static_cast<int64_t>(remaining_layers) * input;   // the later layers' inputs
  int64_t take;
  uint32_t flags;
  if (slot->cursor + full + reserve <= slot->capacity) {
    take = full;
    flags = 0;
  } else if (slot->cursor + input + reserve <= slot->capacity) {
    take = input;
    flags = MOE_SAVE_INPUT_ONLY;
  } else {
    return MOE_ERR_CAPACITY;
  }
  slot->offset[slot->layers] = slot->cursor;
  slot->flags[slot->layers] = flags;
  slot->layers += 1;
  *offset = slot->cursor;
  *forward_flags = flags;
  slot->cursor += take;
  return MOE_OK;
}

moe_status moe_slot_pop(moe_slot* slot, int64_t offset) {
  if (!slot || slot->layers < 1 || slot->layers > MOE_SLOT_MAX_LAYERS) return MOE_ERR_INVALID_ARG;
  if (slot->offset[slot->layers - 1] != offset) return MOE_ERR_INVALID_ARG;   // not the most recent push
  slot->layers -= 1;
  slot->cursor = offset;
  return MOE_OK;
}

size_t moe_ctx_scratch_bytes(const moe_config* cfg) { return config_ok(cfg) ? scratch_layout(cfg).total : 0; }

moe_status moe_ctx_create(const moe_config* cfg, moe_ctx** out) {
  if (!out || !config_ok(cfg)) return MOE_ERR_INVALID_ARG;
  if ((cfg->flags & MOE_REPLAY) && !(cfg->flags & MOE_TRAINING)) return MOE_ERR_INVALID_ARG;
  if (!config_tileable(cfg)) return MOE_ERR_UNSUPPORTED;
  if (cfg->precision == MOE_NVFP4 && (cfg->flags & (MOE_TRAINING | MOE_REPLAY | MOE_POST_NORM)))
    return MOE_ERR_UNSUPPORTED;   // an inference format
  if (!encode_fn()) return MOE_ERR_CUDA;
  moe_ctx* c = new moe_ctx();
  c->cfg = *cfg;
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
    delete c;
    return MOE_ERR_CUDA;
  }
  c->r_cap = row_cap(cfg);
  c->b_cap = block_cap(cfg);
  // BF16 only: MXFP8 pair tiles, single-buffered and bound by their operand
  // loads, measured no faster than two row-block tiles
  c->pair_tiles_auto = cfg->precision == MOE_BF16 &&
                       static_cast<int64_t>(cfg->max_tokens) * cfg->top_k >= 128LL * cfg->num_experts;
  // dense enough for pairs: CTA pairs (one 256 x 256 MMA over two SMs, each
  // loading half the operands, in two-K-chunk stages).  Measured against row
  // blocks in MXFP8 (E = 128 / 96 / 64 / 48 at T = 2048, K = 6, D = 7168:
  // -10 / -4 / +18 / +2 %; a lone block costs a pair twice the SM time) and
  // against one-CTA pairs in BF16 (128 and 192 routes per expert: +2, +6 %).
  c->cta_pairs_auto = static_cast<int64_t>(cfg->max_tokens) * cfg->top_k >=
                      (cfg->precision == MOE_MXFP8 ? 192LL : 128LL) * cfg->num_experts;
  const ScratchLayout L = scratch_layout(cfg);
  c->bytes = L.total;
  if (cudaMalloc(&c->base, c->bytes) != cudaSuccess) {
    delete c;
    return MOE_ERR_CUDA;
  }
  if (cudaMemset(c->base, 0, c->bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(c->base);
    delete c;
    return MOE_ERR_CUDA;
  }
  for (int i = 0; i < MOE_BUF_NUM; ++i) {
    c->buf[i] = L.size[i] ? c->base + L.off[i] : nullptr;
    c->buf_bytes[i] = L.size[i];
  }
  c->err = reinterpret_cast<uint32_t*>(c->buf[MOE_BUF_ERROR]);
  c->clip = reinterpret_cast<unsigned long long*>(B(c, MOE_BUF_ERROR) + 16);
  *out = c;
  return MOE_OK;
}

moe_status moe_ctx_enable_stage_timing(moe_ctx* ctx, int enable) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (enable && !ctx->events) {
    for (int p = 0; p < 2; ++p)
      for (int i = 0; i < 8; ++i) MOE_TRY(cudaEventCreate(&ctx->ev[p][i]));
    ctx->events = true;
  }
  // disabling only stops the recording: a graph captured with timing on
  // still records into these events, so they live until moe_ctx_destroy
  ctx->timing = enable != 0;
  return MOE_OK;
}

moe_status moe_ctx_stage_times(moe_ctx* ctx, int pass, float* ms, int n) {
  if (!ctx || !ms || pass < 0 || pass > 1 || !ctx->events) return MOE_ERR_INVALID_ARG;
  const int stages = pass == 0 ? MOE_FWD_STAGES : MOE_BWD_STAGES;
  if (n < stages) return MOE_ERR_INVALID_ARG;
  MOE_TRY(cudaEventSynchronize(ctx->ev[pass][stages]));
  for (int i = 0; i < stages; ++i) MOE_TRY(cudaEventElapsedTime(&ms[i], ctx->ev[pass][i], ctx->ev[pass][i + 1]));
  return MOE_OK;
}

uint64_t moe_ctx_launch_count(const moe_ctx* ctx) { return ctx ? ctx->launches : 0; }

moe_status moe_ctx_set_post_norm(moe_ctx* ctx, const void* gamma, float eps) {
  if (!ctx || !gamma || !aligned16(gamma) || !(eps > 0.0f) || eps > 3.0e38f) return MOE_ERR_INVALID_ARG;
  if (!(ctx->cfg.flags & MOE_POST_NORM)) return MOE_ERR_INVALID_ARG;
  ctx->norm_gamma = gamma;
  ctx->norm_eps = eps;
  return MOE_OK;
}

moe_status moe_post_norm_backward(moe_ctx* ctx, const void* saved, const void* dout, void* dx_pre, float* dgamma,
                                  cudaStream_t stream) {
  if (!ctx || !saved || !dout || !dx_pre || !dgamma) return MOE_ERR_INVALID_ARG;
  const moe_config& c = ctx->cfg;
  if (!(c.flags & MOE_TRAINING) || !(c.flags & MOE_POST_NORM) || !ctx->norm_gamma) return MOE_ERR_INVALID_ARG;
  if (!aligned16(saved) || !aligned16(dout) || !aligned16(dx_pre) || !aligned16(dgamma)) return MOE_ERR_INVALID_ARG;
  const SavedLayout SL = saved_layout(&c);
  const uint8_t* sv = static_cast<const uint8_t*>(saved);
  const int* hdr = reinterpret_cast<const int*>(sv + SL.off[MOE_SAVED_HEADER]);
  float* nb = reinterpret_cast<float*>(B(ctx, MOE_BUF_NORM));
  const int sms = ctx->max_ctas > 0 ? std::min(ctx->max_ctas, ctx->num_sms) : ctx->num_sms;
  MOE_TRY(launch_post_norm_backward(sv + SL.off[MOE_SAVED_PRENORM], ctx->norm_gamma, dout, c.d_model, ctx->norm_eps,
                                    dx_pre, nb, nb + c.max_tokens, dgamma, c.max_tokens, sms, stream, hdr));
  ctx->launches += 3;
  return MOE_OK;
}

moe_status moe_ctx_test_fused_stall(moe_ctx* ctx, int stall, int64_t wait_cycles) {
  if (!ctx || wait_cycles < 0) return MOE_ERR_INVALID_ARG;
  ctx->fused_stall = stall ? 1 : 0;
  ctx->fused_wait = wait_cycles;
  return MOE_OK;
}

moe_status moe_ctx_test_tile_mode(moe_ctx* ctx, int mode) {
  if (!ctx || mode < 0 || mode > 3) return MOE_ERR_INVALID_ARG;
  ctx->tile_mode = mode;
  return MOE_OK;
}

moe_status moe_ctx_set_max_ctas(moe_ctx* ctx, int max_ctas) {
  if (!ctx || max_ctas < 0) return MOE_ERR_INVALID_ARG;
  ctx->max_ctas = max_ctas;
  return MOE_OK;
}

moe_status moe_ctx_destroy(moe_ctx* ctx) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (ctx->events) {
    for (int p = 0; p < 2; ++p)
      for (int i = 0; i < 8; ++i) cudaEventDestroy(ctx->ev[p][i]);
  }
  const cudaError_t e = cudaFree(ctx->base);
  delete ctx;
  return cuda_status(e);
}

moe_status moe_ctx_buffer(moe_ctx* ctx, int which, void** dev_ptr, size_t* bytes) {
  if (!ctx || which < 0 || which >= MOE_BUF_NUM || !dev_ptr || !bytes) return MOE_ERR_INVALID_ARG;
  *dev_ptr = ctx->buf[which];
  *bytes = ctx->buf_bytes[which];
  return MOE_OK;
}

moe_status moe_ctx_get_error(moe_ctx* ctx, uint32_t* bits) {
  if (!ctx || !bits) return MOE_ERR_INVALID_ARG;
  MOE_TRY(cudaDeviceSynchronize());
  MOE_TRY(cudaMemcpy(bits, ctx->err, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  MOE_TRY(cudaMemset(ctx->err, 0, sizeof(uint32_t)));
  MOE_TRY(cudaDeviceSynchronize());
  return MOE_OK;
}

moe_status moe_ctx_clip_stats(moe_ctx* ctx, uint64_t* counts) {
  if (!ctx || !counts) return MOE_ERR_INVALID_ARG;
  MOE_TRY(cudaDeviceSynchronize());
  MOE_TRY(cudaMemcpy(counts, ctx->clip, 2 * sizeof(uint64_t), cudaMemcpyDeviceToHost));
  MOE_TRY(cudaMemset(ctx->clip, 0, 2 * sizeof(uint64_t)));
  MOE_TRY(cudaDeviceSynchronize());
  return MOE_OK;
}

moe_status moe_debug_copy_to_host(void* host_dst, const void* dev_src, size_t bytes) {
  if (!host_dst || !dev_src) return MOE_ERR_INVALID_ARG;
  MOE_TRY(cudaDeviceSynchronize());
  MOE_TRY(cudaMemcpy(host_dst, dev_src, bytes, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status moe_weight_bytes(moe_precision precision, int32_t E, int32_t N, int32_t K, int with_transpose,
                            size_t* bytes) {
  if (!bytes || E < 1 || N < 32 || K < 32 || N % 32 || K % 32) return MOE_ERR_INVALID_ARG;
  const size_t e = static_cast<size_t>(E), n = static_cast<size_t>(N), k = static_cast<size_t>(K);
  bytes[0] = bytes[1] = bytes[2] = bytes[3] = 0;
  if (precision == MOE_MXFP8 || precision == MOE_MXFP8_1X32) {
    if (N % 128 || K % 128 || (precision == MOE_MXFP8_1X32 && with_transpose) || with_transpose < 0 ||
        with_transpose > 2)
      return MOE_ERR_INVALID_ARG;
    bytes[0] = e * n * k;
    bytes[1] = e * n * (k / 32) + 16;
    if (with_transpose) {
      bytes[2] = with_transpose == 1 ? e * k * n : 0;   // 2: scales only (MN-major input gradients)
      bytes[3] = e * k * (n / 32) + 16;
    }
    return MOE_OK;
  }
  if (precision == MOE_NVFP4) {
    if (N % 128 || K % 64 || with_transpose) return MOE_ERR_INVALID_ARG;
    bytes[0] = nvfp4_chunk_bytes(static_cast<long long>(e * n / 128), K);
    bytes[1] = e * n * sizeof(float);
    return MOE_OK;
  }
  if (precision == MOE_BF16) {
    if (with_transpose < 0 || with_transpose > 1) return MOE_ERR_INVALID_ARG;
    bytes[0] = e * n * k * 2;
    if (with_transpose) bytes[2] = e * k * n * 2;
    return MOE_OK;
  }
  return MOE_ERR_INVALID_ARG;
}

moe_status prepare_block_scaled_weight(const void* w, int32_t E, int32_t N, int32_t K, moe_precision precision,
                                       void* data, uint8_t* scale, void* data_t, uint8_t* scale_t,
                                       cudaStream_t stream) {
  if (!w || !aligned16(w) || E < 1 || N < 32 || K < 32 || N % 32 || K % 32) return MOE_ERR_INVALID_ARG;
  if (precision == MOE_MXFP8_1X32) {
    if (N % 128 || K % 128 || !data || !scale || !aligned16(data) || data_t || scale_t) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_prep_mx_weight_row32(w, E, N, K, static_cast<uint8_t*>(data), scale, stream));
  }
  if (precision == MOE_MXFP8) {
    if (N % 128 || K % 128 || !data || !scale || !aligned16(data)) return MOE_ERR_INVALID_ARG;
    if (data_t && !scale_t) return MOE_ERR_INVALID_ARG;   // transposed codes come with their scales
    if (data_t && !aligned16(data_t)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_prep_mx_weight(w, E, N, K, static_cast<uint8_t*>(data), scale,
                                             static_cast<uint8_t*>(data_t), scale_t, stream));
  }
  if (precision == MOE_NVFP4) {
    if (N % 128 || K % 64 || !data || !scale || !aligned16(data) || !aligned16(scale) || data_t || scale_t)
      return MOE_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    MOE_TRY(cudaGetDevice(&dev));
    MOE_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    return cuda_status(launch_nvfp4_prep_weight(w, E, N, K, static_cast<uint8_t*>(data), reinterpret_cast<float*>(scale),
                                                sms, stream));
  }
  if (precision == MOE_BF16) {
    if (data || scale || scale_t || !data_t || !aligned16(data_t)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_transpose_bf16(w, E, N, K, data_t, stream));
  }
  return MOE_ERR_INVALID_ARG;
}

moe_status moe_forward(moe_ctx* ctx, int32_t T, const void* x, const int32_t* topk_ids, const float* topk_scores,
                       const moe_weight* W13, const moe_weight* W2, void* out, void* saved, uint32_t call_flags,
                       cudaStream_t stream) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  const moe_config& c = ctx->cfg;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T > c.max_tokens) return MOE_ERR_CAPACITY;
  const int D = c.d_model, F = c.d_ff, E = c.num_experts, K = c.top_k;
  const bool train = saved != nullptr;
  if (train && !(c.flags & MOE_TRAINING)) return MOE_ERR_INVALID_ARG;
  if (!weight_ok(W13, c.precision, E, 2 * F, D, false) || !weight_ok(W2, c.precision, E, D, F, false))
    return MOE_ERR_INVALID_ARG;
  if (call_flags & ~(MOE_ACCUMULATE_OUT | MOE_SAVE_INPUT_ONLY | MOE_FUSED_LAUNCH)) return MOE_ERR_INVALID_ARG;
  const bool fused = (call_flags & MOE_FUSED_LAUNCH) != 0;
  if (fused) {
    const int64_t tk = static_cast<int64_t>(T) * K;
    const int64_t max_blocks = tk / 128 + std::min<int64_t>(E, tk) + 1;
    if (train || c.precision != MOE_MXFP8 || (c.flags & MOE_POST_NORM) || pair_tiles(D) != 2 ||
        tk > kFusedMaxRoutes || max_blocks >= 1024 || !ctx->buf[MOE_BUF_SYNC])
      return MOE_ERR_UNSUPPORTED;
  }
  const bool input_only = (call_flags & MOE_SAVE_INPUT_ONLY) != 0;
  if (input_only && (!train || !(c.flags & MOE_REPLAY))) return MOE_ERR_INVALID_ARG;
  const bool nvfp4 = c.precision == MOE_NVFP4;   // inference only (no saved state, no single launch)
  if (T == 0) return MOE_OK;
  if (!x || !topk_ids || !topk_scores || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out) || (saved && !aligned16(saved))) return MOE_ERR_INVALID_ARG;
  const bool norm = (c.flags & MOE_POST_NORM) != 0;
  if (norm && !ctx->norm_gamma) return MOE_ERR_INVALID_ARG;

  const SavedLayout SL = saved_layout(&c, input_only);
  uint8_t* sv = static_cast<uint8_t*>(saved);
  if (train) {
    // bounded: a caller cycling through fresh buffers forgets the oldest
    // modes (their backwards are then taken at their word) instead of growing
    if (ctx->saved_input_only.size() >= 4096 && !ctx->saved_input_only.count(saved)) ctx->saved_input_only.clear();
    ctx->saved_input_only[saved] = input_only;
  }
  if (input_only)   // the backward replays from this copy of x
    MOE_TRY(cudaMemcpyAsync(sv + SL.off[MOE_SAVED_X], x, static_cast<size_t>(T) * D * 2, cudaMemcpyDeviceToDevice,
                            stream));
  const RoutingPtrs rp = routing_ptrs(train ? sv : B(ctx, MOE_BUF_ROUTING), SL);
  const int64_t R = ctx->r_cap;
  const int sms = ctx->max_ctas > 0 ? std::min(ctx->max_ctas, ctx->num_sms) : ctx->num_sms;

  MOE_TRY(stage_mark(ctx, 0, 0, stream));
  if (fused) {
    MOE_PASS(run_fused_forward(ctx, T, x, topk_ids, topk_scores, rp, W13, W2, out,
                               (call_flags & MOE_ACCUMULATE_OUT) != 0, sms, stream));
    for (int i = 1; i <= MOE_FWD_STAGES; ++i) MOE_TRY(stage_mark(ctx, 0, i, stream));
    return MOE_OK;
  }
  MOE_TRY(launch_route(topk_ids, topk_scores, T, K, E, static_cast<int>(R), (c.flags & MOE_DEBUG_CHECKS) ? 1 : 0,
                       rp, ctx->err, stream));
  ctx->launches += 1;
  MOE_TRY(stage_mark(ctx, 0, 1, stream));
  uint8_t* act = (train && !input_only) ? sv : nullptr;   // where the expert state is saved
  uint8_t* h3 = act ? act + SL.off[MOE_SAVED_H3] : B(ctx, MOE_BUF_H3);   // saved for the score gradient
  if (nvfp4) {
    MOE_PASS(run_nvfp4(ctx, T, x, rp, W13, W2, sms, stream));
  } else {
    MOE_PASS(run_gather_w13(ctx, x, rp, W13, act, SL, true, sms, stream));
    MOE_PASS(run_w2(ctx, rp, W2, h3, sms, stream));
  }
  MOE_TRY(stage_mark(ctx, 0, 4, stream));

  // ---- combine
  MOE_TRY(launch_combine(h3, D, K, rp.inv, rp.scores, out, T, (call_flags & MOE_ACCUMULATE_OUT) != 0, sms, stream,
                         nullptr, norm ? ctx->norm_gamma : nullptr, ctx->norm_eps,
                         (norm && train) ? sv + SL.off[MOE_SAVED_PRENORM] : nullptr));
  ctx->launches += 1;
  MOE_TRY(stage_mark(ctx, 0, 5, stream));
  return MOE_OK;
}

moe_status moe_backward(moe_ctx* ctx, const void* saved, const void* dout, const moe_weight* W13,
                        const moe_weight* W2, void* dx, void* dW13, void* dW2, float* d_scores, uint32_t call_flags,
                        cudaStream_t stream) {
  if (!ctx || !saved || !dout || !dx || !dW13 || !dW2) return MOE_ERR_INVALID_ARG;
  const moe_config& c = ctx->cfg;
  if (!(c.flags & MOE_TRAINING)) return MOE_ERR_INVALID_ARG;
  const int D = c.d_model, F = c.d_ff, E = c.num_experts, K = c.top_k;
  const bool mx = c.precision == MOE_MXFP8;
  if (!weight_ok(W13, c.precision, E, 2 * F, D, true) || !weight_ok(W2, c.precision, E, D, F, true))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(saved) || !aligned16(dout) || !aligned16(dx) || !aligned16(dW13) || !aligned16(dW2))
    return MOE_ERR_INVALID_ARG;
  if (call_flags & ~(MOE_ACCUMULATE_DX | MOE_DW_FP32 | MOE_DW_ACCUMULATE | MOE_REPLAY_FORWARD))
    return MOE_ERR_INVALID_ARG;
  const bool replay = (call_flags & MOE_REPLAY_FORWARD) != 0;
  if (replay && !(c.flags & MOE_REPLAY)) return MOE_ERR_INVALID_ARG;
  const auto known = ctx->saved_input_only.find(saved);
  if (known != ctx->saved_input_only.end() && known->second != replay) return MOE_ERR_INVALID_ARG;

  const SavedLayout SL = saved_layout(&c);   // the expert-state fields (in `sa`)
  uint8_t* sv = static_cast<uint8_t*>(const_cast<void*>(saved));
  const RoutingPtrs rp = routing_ptrs(sv, SL);   // same offsets in an input-only state
  const int64_t R = ctx->r_cap;
  const int sms = ctx->max_ctas > 0 ? std::min(ctx->max_ctas, ctx->num_sms) : ctx->num_sms;
  const int dw_fp32 = (call_flags & MOE_DW_FP32) ? 1 : 0;
  const int dw_acc = (call_flags & MOE_DW_ACCUMULATE) ? 1 : 0;
  // dW leaves through shared memory and TMA, except a BF16 accumulation
  // (which rounds old + new once, in the epilogue)
  const int dw_store = dw_fp32 ? (dw_acc ? kDwAddF32 : kDwStoreF32) : (dw_acc ? kDwDirect : kDwStoreBf16);

  // ---- replay: rebuild the expert state of an input-only forward from its
  // saved x and routing, with the forward's own kernels, in the context's
  // replay scratch ([DM] section 04: the backward republishes x and rebuilds
  // the expert state in scratch)
  uint8_t* sa = sv;
  if (replay) {
    sa = B(ctx, MOE_BUF_REPLAY);
    const SavedLayout SI = saved_layout(&c, true);
    MOE_PASS(run_gather_w13(ctx, sv + SI.off[MOE_SAVED_X], rp, W13, sa, SL, false, sms, stream));
    if (d_scores) MOE_PASS(run_w2(ctx, rp, W2, sa + SL.off[MOE_SAVED_H3], sms, stream));
  }

  // ---- dh3 = s * dY: row bundle (W2 DGRAD) and column bundle (W2 WGRAD)
  MOE_TRY(stage_mark(ctx, 1, 0, stream));
  CUtensorMap tr, tc;
  if (mx && (!make_tmap(&tr, B(ctx, MOE_BUF_DH3ROW), true, R, D, 128) ||
             !make_tmap(&tc, B(ctx, MOE_BUF_DH3COL), true, D, R, 128)))
    return MOE_ERR_CUDA;
  MOE_TRY(launch_gather_both(mx, true, dout, D, K, rp, B(ctx, MOE_BUF_DH3ROW), B(ctx, MOE_BUF_DH3ROW_SCALE),
                             B(ctx, MOE_BUF_DH3COL), B(ctx, MOE_BUF_DH3COL_SCALE), static_cast<int>(R),
                             static_cast<int>(ctx->b_cap), sms, stream, &tr, &tc));
  ctx->launches += 1;
  MOE_TRY(stage_mark(ctx, 1, 1, stream));

  // ---- W2 DGRAD + SwiGLU backward -> dh1 row and column bundles
  GemmLaunch g1{};
  g1.mx = mx;
  g1.na = 1;   // the SwiGLU-backward epilogue needs two accumulator buffers
  g1.epi = kEpiSwigluBwd;
  // over row-block pairs in BF16 only: a 256-wide MXFP8 accumulator is
  // single-buffered, and this epilogue reads it to the end of its work.
  // BF16 contexts whose forward runs on CTA pairs run this GEMM on them too
  // (256-feature cluster tiles).
  const bool cta1 = !mx && forward_tiles(ctx) == kGroupedMC && F % 256 == 0;
  g1.mode = cta1 ? kGroupedMC : ((use_pairs(ctx) && !mx) ? kGroupedMP : kGroupedM);
  // MXFP8 weights prepared without transposed codes: A is W2's forward codes
  // [E*D rows (K), F columns (M)], read MN-major
  const bool mn2 = mx && W2->data_t == nullptr;
  if (!(mn2 ? make_tmap(&g1.tmA, W2->data, mx, static_cast<int64_t>(E) * D, F, 128)
            : make_tmap(&g1.tmA, W2->data_t, mx, static_cast<int64_t>(E) * F, D, 128)) ||
      !make_tmap(&g1.tmB, B(ctx, MOE_BUF_DH3ROW), mx, R, D, 32) ||
      !make_grouped_m_boxes(&g1, mn2 ? W2->data : W2->data_t, static_cast<int64_t>(E) * F, W2->scale_t,
                            B(ctx, MOE_BUF_DH3ROW), R, mx, D))
    return MOE_ERR_CUDA;
  g1.p.a_mn = mn2 ? 1 : 0;
  GemmParams& p1 = g1.p;
  p1.hdr = rp.hdr;
  p1.blocks = rp.blocks;
  p1.poffsets = rp.poffsets;
  p1.E = E;
  p1.b_box_rows = 32;
  p1.n_tiles = F / (cta1 ? 256 : 128 * g1.na);
  p1.K = D;
  p1.a_rows_per_expert = F;
  p1.sfa = W2->scale_t;
  p1.sfa_ts = D / 128;
  p1.sfb = B(ctx, MOE_BUF_DH3ROW_SCALE);
  p1.sfb_ts = D / 128;
  p1.h1 = reinterpret_cast<__nv_bfloat16*>(sa + SL.off[MOE_SAVED_H1]);
  p1.h1_pitch = 2 * F;
  p1.out0 = B(ctx, MOE_BUF_DH1ROW);
  p1.out0_pitch = 2 * F;
  p1.out0_sf = B(ctx, MOE_BUF_DH1ROW_SCALE);
  p1.out0_sf_kg = 2 * F / 128;
  p1.out1 = B(ctx, MOE_BUF_DH1COL);
  p1.out1_pitch = R;
  p1.out1_sf = B(ctx, MOE_BUF_DH1COL_SCALE);
  p1.b_cap = static_cast<int>(ctx->b_cap);
  p1.F = F;
  p1.swiglu_limit = c.swiglu_limit;
  p1.err = ctx->err;
  g1.max_tiles = static_cast<int>(ctx->b_cap * p1.n_tiles);
  MOE_TRY(launch_gemm(g1, sms, stream));
  ctx->launches += 1;
  MOE_TRY(stage_mark(ctx, 1, 2, stream));

  // ---- W2 WGRAD: dW2[e] = dh3_e^T h2_e   ([D, F] per expert)
  GemmLaunch g2{};
  g2.mx = mx;
  g2.na = 1;
  g2.epi = kEpiWgrad;
  g2.mode = kGroupedK;
  if (!make_tmap(&g2.tmA, B(ctx, MOE_BUF_DH3COL), mx, D, R, 128) ||
      !make_tmap(&g2.tmB, sa + SL.off[MOE_SAVED_H2COL], mx, F, R, 128) ||
      !make_narrow_tmaps(&g2, B(ctx, MOE_BUF_DH3COL), D, sa + SL.off[MOE_SAVED_H2COL], F, mx, R))
    return MOE_ERR_CUDA;
  GemmParams& p2 = g2.p;
  p2.hdr = rp.hdr;
  p2.blocks = rp.blocks;
  p2.poffsets = rp.poffsets;
  p2.E = E;
  p2.b_box_rows = 128;
  p2.m_tiles = D / 128;
  p2.n_tiles = F / 128;
  p2.bstart = rp.bstart;
  p2.sfa = B(ctx, MOE_BUF_DH3COL_SCALE);
  p2.sfa_ts = ctx->b_cap;
  p2.sfb = mx ? sa + SL.off[MOE_SAVED_H2COL_SCALE] : nullptr;
  p2.sfb_ts = ctx->b_cap;
  p2.out0 = dW2;
  p2.out0_pitch = F;
  p2.dw_fp32 = dw_fp32;
  p2.dw_accum = dw_acc;
  p2.tma_store = dw_store;
  if (dw_store != kDwDirect && !make_out_tmap(&g2.tmC, dW2, static_cast<int64_t>(E) * D, F, dw_fp32 != 0)) return MOE_ERR_CUDA;
  p2.err = ctx->err;
  g2.max_tiles = E * (D / 128) * (F / 128);
  MOE_TRY(launch_gemm(g2, sms, stream));
  ctx->launches += 1;
  MOE_TRY(stage_mark(ctx, 1, 3, stream));

  // ---- W13 DGRAD: dxr = dh1 W13[e]
  GemmLaunch g3{};
  const bool pairs3 = use_pairs(ctx);
  // BF16 on CTA pairs as its forward (256-feature cluster tiles of D)
  const bool cta3 = !mx && forward_tiles(ctx) == kGroupedMC && D % 256 == 0;
  g3.mx = mx;
  g3.na = (pairs3 || cta3) ? 1 : pair_tiles(D);
  g3.epi = kEpiStore;
  g3.mode = cta3 ? kGroupedMC : (pairs3 ? kGroupedMP : kGroupedM);
  // MXFP8 without transposed codes: A is W13's forward codes [E*2F rows (K),
  // D columns (M)], read MN-major, one box per 128-column weight tile
  const bool mn13 = mx && W13->data_t == nullptr;
  if (!(mn13 ? make_tmap(&g3.tmA, W13->data, mx, static_cast<int64_t>(E) * 2 * F, D, 128)
             : make_tmap(&g3.tmA, W13->data_t, mx, static_cast<int64_t>(E) * D, 2 * F, 128)) ||
      !make_tmap(&g3.tmB, B(ctx, MOE_BUF_DH1ROW), mx, R, 2 * F, 32) ||
      !make_grouped_m_boxes(&g3, mn13 ? W13->data : W13->data_t, static_cast<int64_t>(E) * D, W13->scale_t,
                            B(ctx, MOE_BUF_DH1ROW), R, mx, 2 * F))
    return MOE_ERR_CUDA;
  if (mn13) {
    g3.p.a_mn = 1;
    g3.p.a_pair_box = 0;   // one box and one scale atom per weight tile
  }
  GemmParams& p3 = g3.p;
  p3.hdr = rp.hdr;
  p3.blocks = rp.blocks;
  p3.poffsets = rp.poffsets;
  p3.E = E;
  p3.b_box_rows = 32;
  p3.n_tiles = D / (cta3 ? 256 : 128 * g3.na);
  p3.K = 2 * F;
  p3.a_rows_per_expert = D;
  p3.sfa = W13->scale_t;
  p3.sfa_ts = 2 * F / 128;
  p3.sfb = B(ctx, MOE_BUF_DH1ROW_SCALE);
  p3.sfb_ts = 2 * F / 128;
  p3.out0 = B(ctx, MOE_BUF_DXR);
  p3.out0_pitch = D;
  p3.F = F;
  p3.err = ctx->err;
  g3.max_tiles = static_cast<int>(ctx->b_cap * p3.n_tiles);
  MOE_TRY(launch_gemm(g3, sms, stream));
  ctx->launches += 1;
  MOE_TRY(stage_mark(ctx, 1, 4, stream));

  // ---- W13 WGRAD: dW13[e] = dh1_e^T x_e   ([2F, D] per expert)
  GemmLaunch g4{};
  g4.mx = mx;
  g4.na = 1;
  g4.epi = kEpiWgrad;
  g4.mode = kGroupedK;
  if (!make_tmap(&g4.tmA, B(ctx, MOE_BUF_DH1COL), mx, 2 * F, R, 128) ||
      !make_tmap(&g4.tmB, sa + SL.off[MOE_SAVED_XCOL], mx, D, R, 128) ||
      !make_narrow_tmaps(&g4, B(ctx, MOE_BUF_DH1COL), 2 * F, sa + SL.off[MOE_SAVED_XCOL], D, mx, R))
    return MOE_ERR_CUDA;
  GemmParams& p4 = g4.p;
  p4.hdr = rp.hdr;
  p4.blocks = rp.blocks;
  p4.poffsets = rp.poffsets;
  p4.E = E;
  p4.b_box_rows = 128;
  p4.m_tiles = 2 * F / 128;
  p4.n_tiles = D / 128;
  p4.bstart = rp.bstart;
  p4.sfa = B(ctx, MOE_BUF_DH1COL_SCALE);
  p4.sfa_ts = ctx->b_cap;
  p4.sfb = mx ? sa + SL.off[MOE_SAVED_XCOL_SCALE] : nullptr;
  p4.sfb_ts = ctx->b_cap;
  p4.out0 = dW13;
  p4.out0_pitch = D;
  p4.dw_fp32 = dw_fp32;
  p4.dw_accum = dw_acc;
  p4.tma_store = dw_store;
  if (dw_store != kDwDirect && !make_out_tmap(&g4.tmC, dW13, static_cast<int64_t>(E) * 2 * F, D, dw_fp32 != 0)) return MOE_ERR_CUDA;
  p4.err = ctx->err;
  g4.max_tiles = E * (2 * F / 128) * (D / 128);
  MOE_TRY(launch_gemm(g4, sms, stream));
  ctx->launches += 1;
  MOE_TRY(stage_mark(ctx, 1, 5, stream));

  // ---- dX[t] = sum_k dxr(t,k)
  MOE_TRY(launch_combine(B(ctx, MOE_BUF_DXR), D, K, rp.inv, nullptr, dx, c.max_tokens,
                         (call_flags & MOE_ACCUMULATE_DX) != 0, sms, stream, rp.hdr));
  ctx->launches += 1;
  MOE_TRY(stage_mark(ctx, 1, 6, stream));
  if (d_scores) {
    MOE_TRY(launch_score_grad(sa + SL.off[MOE_SAVED_H3], dout, D, K, rp.inv, d_scores, c.max_tokens, sms, stream,
                              rp.hdr));
    ctx->launches += 1;
  }
  return MOE_OK;
}

}  // extern "C"
