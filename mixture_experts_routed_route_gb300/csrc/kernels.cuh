// Launch interface of the MoE kernels (internal to the library).
#pragma once

#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace moe {

// ------------------------------------------------ per-device kernel set-up

// Devices a process may drive (device ordinals 0 .. kMaxDevices - 1).
constexpr int kMaxDevices = 64;

// A kernel attribute such as the dynamic shared-memory opt-in belongs to
// the context of the device that was current when it was set, so each
// device needs its own set-up.  once() runs `fn` the first time it is
// called with a device current, under a lock (host threads may race on
// the first launch), and remembers success per device; a failed set-up is
// tried again on the next call.
struct PerDeviceOnce {
  std::atomic<int> done[kMaxDevices] = {};
  std::mutex mu;

  template <typename Fn>
  cudaError_t once(Fn&& fn) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lk(mu);
    if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    e = fn();
    if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
    return e;
  }
};

// Device view of one routing state (the saved-state prefix or the
// context's inference copy).  Layout and meaning of every array are those of
// moe_saved_field in moe_gb300.h.
struct RoutingPtrs {
  int* hdr;       // [0] T, [1] blocks, [2] padded rows used, [3] active routes
  int* counts;    // [E]
  int* offsets;   // [E+1]
  int* poffsets;  // [E+1]
  int* perm;      // [r_cap]
  int* inv;       // [T_max*K]
  int4* blocks;   // [b_cap] (expert, first row, rows, 0)
  float* scores;  // [T_max*K]
  int* bstart;    // [E+1] first row block of each expert
  int* row_block; // [r_cap/32] row block of each 32-row group
};

// MXFP8 scale atoms: 128 operand rows x 4 consecutive 32-value blocks, 512
// bytes, row p / block l at byte (p % 32) * 16 + (p / 32) * 4 + l (the order
// tcgen05.cp 32x128b.warpx4 lays scales into tensor memory).
__host__ __device__ __forceinline__ long long sf_atom_byte(int p, int l) {
  return (p & 31) * 16 + (p >> 5) * 4 + l;
}

constexpr int kPad = 32;        // rows of every expert are padded to this
constexpr int kBlockRows = 128; // rows per GEMM row block (MMA N <= 128)

cudaError_t launch_route(const int32_t* ids, const float* scores, int T, int K, int E, int r_cap, int debug,
                         const RoutingPtrs& rp, uint32_t* err, cudaStream_t stream);

// Row bundle: dst[r] = q(s * src[perm[r] / K]) for every used row r (s = the
// route's score when `use_scores`, else 1; zero rows for padding).
cudaError_t launch_gather_rows(bool mx, bool use_scores, const void* src, int D, int K, const RoutingPtrs& rp,
                               void* dst, uint8_t* dst_sf, int r_cap, int num_sms, cudaStream_t stream);

// Row bundle and column bundle of the same gathered rows in one pass
// (training): dstT[d][r] holds the rows transposed to [D, r_cap]; MXFP8
// quantises it along rows in 32-row blocks (WGRAD contracts over rows).
// MXFP8 needs tm_row / tm_col: 128 x 128-byte boxes, 128-byte swizzle, over
// dst [r_cap, D] and dstT [D, r_cap] (the bundles leave by TMA store).
cudaError_t launch_gather_both(bool mx, bool use_scores, const void* src, int D, int K, const RoutingPtrs& rp,
                               void* dst, uint8_t* dst_sf, void* dstT, uint8_t* dstT_sf, int r_cap, int b_cap,
                               int num_sms, cudaStream_t stream, const CUtensorMap* tm_row = nullptr,
                               const CUtensorMap* tm_col = nullptr);

// out[t] = bf16((accumulate ? out[t] : 0) + sum_k s(t,k) * h[inv(t,k)]),
// FP32, k in order; s = 1 when `scores` is NULL.  The token count is T, or
// hdr[0] (read on the device, at most T) when `hdr` is given.  With `gamma`
// (bf16 [D]) that row x is then normalised: out[t] = bf16(gamma x r),
// r = 1/sqrt(mean x^2 + eps); x is kept in `xsave` (bf16 [T, D]) if given.
cudaError_t launch_combine(const void* h, int D, int K, const int* inv, const float* scores, void* out, int T,
                           bool accumulate, int num_sms, cudaStream_t stream, const int* hdr = nullptr,
                           const void* gamma = nullptr, float eps = 0.0f, void* xsave = nullptr);

// Tokens per dgamma partial sum of the post-norm backward.
constexpr int kPostNormSlab = 64;

// Post-norm backward for tokens t < min(T, hdr[0]): dx = bf16(r g - x r^3 c)
// with g = gamma dy, c = mean_d(g x), r from x (also written to rstd[T]);
// dgamma[d] = sum_t dy x r through partial[ceil(T/kPostNormSlab)][D] slab sums.
cudaError_t launch_post_norm_backward(const void* x, const void* gamma, const void* dy, int D, float eps, void* dx,
                                      float* rstd, float* partial, float* dgamma, int T, int num_sms,
                                      cudaStream_t stream, const int* hdr);

// dp[t*K+k] = <h3[inv(t,k)], dY[t]> in FP32 (fixed order), 0 if inactive;
// tokens t < min(T, hdr[0]).
cudaError_t launch_score_grad(const void* h3, const void* dY, int D, int K, const int* inv, float* dp, int T,
                              int num_sms, cudaStream_t stream, const int* hdr);

cudaError_t launch_prep_mx_weight(const void* w, int E, int N, int K, uint8_t* q, uint8_t* sf, uint8_t* qT,
                                  uint8_t* sfT, cudaStream_t stream);
// 1x32 blocks along K (inference weights): codes [E,N,K] and scale atoms
// [E*N/128][K/128], no transposed copy.
cudaError_t launch_prep_mx_weight_row32(const void* w, int E, int N, int K, uint8_t* q, uint8_t* sf,
                                        cudaStream_t stream);
cudaError_t launch_transpose_bf16(const void* w, int E, int N, int K, void* wT, cudaStream_t stream);

// ------------------------------------------------------------------ NVFP4
// (nvfp4.cu: format, chunk layout and GEMM design.)  Chunks are 128 rows x
// 64 values of one operand: 4096 code bytes, then 512 block-scale bytes.

// Bytes of the chunks of `row_tiles` 128-row tiles with K values per row.
size_t nvfp4_chunk_bytes(long long row_tiles, int K);

// Weight [E, N, K] BF16 -> chunks of its row tiles and FP32 row scales g
// [E*N]; N % 128 == 0, K % 64 == 0.
cudaError_t launch_nvfp4_prep_weight(const void* w, int E, int N, int K, uint8_t* chunks, float* g, int num_sms,
                                     cudaStream_t stream);

// Routed rows r < hdr[2] -> chunks of their routing blocks and g [r_cap]:
// BF16 x[perm[r] / top_k] (zeros for pad rows) or, with f32_rows, the FP32
// rows src[r] ([r_cap, K]).
cudaError_t launch_nvfp4_rows(bool f32_rows, const void* src, int K, int top_k, const RoutingPtrs& rp, int r_cap,
                              uint8_t* chunks, float* g, int num_sms, cudaStream_t stream);

struct Fp4GemmParams {
  const uint8_t* a;     // weight chunks
  const float* ga;      // weight row scales [E * N]
  const uint8_t* b;     // routed activation chunks (per routing block)
  const float* gb;      // routed row scales [r_cap]
  const int* hdr;       // routing header: hdr[1] routing blocks
  const int4* blocks;   // (expert, first row, rows, -) per routing block
  void* out;            // SwiGLU: FP32 h2 [r_cap, ld]; otherwise BF16 h3 [r_cap, ld]
  int ks;               // K / 64 stages
  int n_tiles;          // 128-wide output slices per routing block (F/128 or D/128)
  int a_tiles_e;        // 128-row weight tiles per expert (2F/128 or D/128)
  int ld;               // output row pitch in elements
  float swiglu_limit;   // clamped SwiGLU (0: plain)
  unsigned long long* clip;   // [2] clamped gate / up counts, or NULL
  uint32_t* err;        // device error word
};

// Grouped-M GEMM over routing blocks x 128-feature slices; swiglu: W13 (gate
// tile n and up tile n + F/128 of the block's expert) with the SwiGLU
// epilogue, else W2 with the BF16 store.  `grid` persistent CTAs.
cudaError_t launch_nvfp4_gemm(const Fp4GemmParams& p, bool swiglu, int grid, cudaStream_t stream);

// ------------------------------------------------------------- grouped GEMM

// kGroupedMP: grouped-M over row-block pairs (B up to 256 rows, one A tile
// of 128 rows per stage; the SwiGLU forward's A tile is 64 gate rows then the
// 64 up rows of the same features).  kGroupedMC: the same tiles on CTA
// pairs (clusters of two): the pair's two CTAs take adjacent A tiles and one
// routing block each of the same row-block pair, and one 256 x 256 MMA
// (cta_group::2) covers both, so each SM loads 128 B rows instead of 256.
enum GemmMode { kGroupedM = 0, kGroupedK = 1, kGroupedMP = 2, kGroupedMC = 3 };
// How a weight-gradient epilogue writes dW: plain stores (BF16 accumulate),
// or staged in shared memory and moved by TMA: a BF16 store, an FP32 store,
// or an FP32 reduce-add into the existing dW (one FP32 add per element,
// formed in L2).
enum DwStore { kDwDirect = 0, kDwStoreBf16 = 1, kDwStoreF32 = 2, kDwAddF32 = 3 };
enum GemmEpi { kEpiSwigluFwd = 0, kEpiStore = 1, kEpiSwigluBwd = 2, kEpiWgrad = 3 };

struct GemmParams {
  // routing
  const int* hdr;
  const int4* blocks;
  const int* poffsets;
  const int* bstart;      // grouped-K: first row block of each expert
  int E;
  int n_tiles;            // grouped-M: 128-wide output tiles per expert; grouped-K: N/128
  int m_tiles;            // grouped-K: M/128
  int K;                  // grouped-M: contraction length
  int a_rows_per_expert;  // grouped-M: rows of A per expert
  int a_up_offset;        // SwiGLU forward: row offset of the up half (F)
  int b_box_rows;         // rows of one B tensor-map box (32, or 128 in grouped-K)
  // MXFP8 scale atoms of the operands (512 bytes each).  Atom of an A tile:
  // grouped-M (A row / 128) * sfa_ts + stage, grouped-K m_tile * sfa_ts +
  // (first block of the expert + stage); B likewise with the row block
  // (grouped-M) or n_tile (grouped-K).
  const uint8_t* sfa;
  long long sfa_ts;
  const uint8_t* sfb;
  long long sfb_ts;
  // epilogue outputs (pitches in elements)
  void* out0;
  long long out0_pitch;
  uint8_t* out0_sf;       // row-bundle scale atoms [b_cap][out0_sf_kg]
  int out0_sf_kg;
  void* out1;
  long long out1_pitch;
  uint8_t* out1_sf;       // column-bundle scale atoms [features/128][b_cap]
  int b_cap;
  __nv_bfloat16* h1;      // SwiGLU forward: written when save_h1; backward: read
  long long h1_pitch;
  int F;
  int save_h1;
  int want_col;
  int dw_fp32;
  int dw_accum;
  int tma_store;          // weight gradient through shared memory + TMA (kDwStore*)
  // grouped-M, both A tiles of a stage in one copy: aux[0] holds their data
  // (1: adjacent 128-row tiles, a 256-row box; 2: gate and up halves F rows
  // apart, a 3D [halves][F][K] box) and aux[2] their two scale atoms (1:
  // adjacent tiles, 3D atom view; 2: halves, 4D atom view)
  int a_pair_box;
  float swiglu_limit;     // SwiGLU epilogues: clamp g <= L and |u| <= L when L > 0
  unsigned long long* clip;  // SwiGLU forward with a limit: [2] counts of clamped g, u (or null)
  int b_full_box;         // grouped-M: aux[1] loads a full 128-row block in one box
  // grouped-M, MXFP8: A is read MN-major from the weight as prepared for the
  // forward (tmA over [E * K rows, M cols], 128 M-bytes x 128 K-rows boxes):
  // the input-gradient GEMMs need no transposed copy of the codes
  int a_mn;
  // Set by the launcher from the grid size: the step of one grid in tile
  // coordinates (tile, n, m, e), by which the producer, MMA and scale-copy
  // roles advance their tiles.
  int walk[4];
  uint32_t* err;
};

struct GemmLaunch {
  bool mx;
  int na;                 // A tiles per stage (gate + up, or two adjacent weight tiles)
  GemmEpi epi;
  GemmMode mode;
  CUtensorMap tmA, tmB, tmC;  // tmC: weight-gradient output (TMA store)
  // auxiliary maps, by mode:
  //  grouped-K: aux[0] / aux[1] = A / B with 64-byte wide boxes (64B swizzle),
  //             aux[2] / aux[3] = A / B with 32-byte wide boxes (32B swizzle),
  //             for a last stage that holds only 64 or 32 bytes of each row;
  //  grouped-M: aux[0] = both A tiles of a stage in one box (a_pair_box),
  //             aux[1] = B with 128-row boxes (b_full_box),
  //             aux[2] = the A tiles' two scale atoms in one box (a_pair_box).
  CUtensorMap aux[4];
  GemmParams p;
  int max_tiles;          // upper bound of the tile count (grid sizing)
};

cudaError_t launch_gemm(const GemmLaunch& g, int num_sms, cudaStream_t stream);

// ------------------------------------------------- single-launch forward
// MXFP8 inference forward in one persistent cooperative grid (fused.cu):
// routing, gather, W13 + SwiGLU, W2, combine, coordinated by counters in
// `sync` ((3 + 2 b_cap) ints, zero before the first launch).

// Largest T*K the single-launch forward takes (the routing runs in one CTA
// and every row block must fit the GEMMs' shared-memory block cache).
constexpr int kFusedMaxRoutes = 1024;

struct FusedArgs {
  const int32_t* ids;
  const float* scores;
  const __nv_bfloat16* x;
  __nv_bfloat16* out;
  int T, K, E, D, F;
  int debug;        // flag ID -1 routes with a nonzero score
  int accumulate;   // out = bf16(out + routed sum)
  RoutingPtrs rp;   // routing arrays, written by CTA 0
  uint8_t* xrow;    // x row bundle [r_cap, D] and its scale atoms [b_cap][D/128]
  uint8_t* xsf;
  int* sync;
  int b_cap;
  long long wait_cycles;   // limit of every counter wait (SM cycles)
  int stall;               // test only: W2 tiles wait for one W13 tile more than exist
  GemmParams g13, g2;      // the two GEMMs (g13.out0 = h2 row bundle, g2.out0 = h3)
};

struct FusedLaunch {
  CUtensorMap a13, sf13, bx32, bx128;   // W13 gate/up box, their atoms, x bundle 32/128-row boxes
  CUtensorMap a2, sf2, bh32, bh128;     // W2 256-row box, its atoms, h2 bundle 32/128-row boxes
  FusedArgs args;
  int max_blocks;   // bound on the routing's row blocks (grid sizing)
};

cudaError_t launch_fused_forward(const FusedLaunch& L, int num_sms, cudaStream_t stream);

// ------------------------------------------------------------- tensor maps
// (host side, tmaps.cu; each returns false when the driver rejects the map)

// The driver's cuTensorMapEncodeTiled, looked up once (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();

// 2D operand map over a row-major [rows, cols] matrix (E4M3 bytes when mx,
// else BF16): boxes `row_bytes` (128, 64 or 32) wide with the matching
// swizzle and `box_rows` tall.
bool make_tmap(CUtensorMap* tm, const void* base, bool mx, int64_t rows, int64_t cols, int box_rows,
               int row_bytes = 128);

// A tensor map of any rank (dims / box innermost first, byte strides of
// dims 1..rank-1), no interleave.
bool make_tmap_nd(CUtensorMap* tm, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
                  const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw);

// Weight tiles per stage of a grouped-M store GEMM with an n-feature output:
// 2 when n is a multiple of 256 (two adjacent tiles share each activation
// box), else 1.
int pair_tiles(int64_t n);

// The narrow-box maps (64- and 32-byte rows) a weight-gradient GEMM uses for
// a short last stage, into g->aux[0..3].
bool make_narrow_tmaps(GemmLaunch* g, const void* a, int64_t a_rows, const void* b, int64_t b_rows, bool mx,
                       int64_t cols);

// The larger boxes of a grouped-M GEMM (both A tiles of a stage in one
// copy, their scale atoms in one copy, a full 128-row block of B in one
// box), into g->aux[0..2]; sets g->p.a_pair_box and g->p.b_full_box.
// `halves_f` = F for W13's gate and up halves, else 0.
bool make_grouped_m_boxes(GemmLaunch* g, const void* a, int64_t a_rows, const void* a_sf, const void* b,
                          int64_t b_rows, bool mx, int64_t cols, int64_t halves_f = 0);

// Output map of a weight gradient [rows, cols], BF16 or FP32: boxes of 128
// bytes (64 BF16 or 32 FP32 columns) x 128 rows in the 128-byte swizzle the
// epilogue stages.
bool make_out_tmap(CUtensorMap* tm, void* base, int64_t rows, int64_t cols, bool fp32 = false);

}  // namespace moe
