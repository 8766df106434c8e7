// Building blocks of the grouped GEMMs on the 5th-generation tensor cores,
// shared by the GEMM kernels (gemm.cu) and the single-launch forward
// (fused.cu): tile decoding over the routing's row blocks, the epilogues
// (SwiGLU forward and backward, BF16 store, weight-gradient staging) and the
// per-configuration shared-memory and tensor-memory plan.  The design notes
// are at the top of gemm.cu.
#pragma once

#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kABytes = 128 * 128;  // one 128-row x 128-byte operand tile
constexpr int kBBytes = 128 * 128;
constexpr int kAtom = 512;          // one scale atom
constexpr int kEpiBarrier = 1;      // named barriers 1, 2: one per epilogue group
// Tile metadata cached in shared memory at kernel start, so no role pays a
// dependent global load per tile: the routing's row blocks (grouped-M, the
// first kCacheBlocks of them) or the experts' row offsets and first blocks
// (grouped-K, E <= 1024).
constexpr int kCacheBlocks = 1024;
constexpr int kCacheBytes = 16384;

struct Tile {
  int e;
  int blk;       // grouped-M: routing row block
  int a_row[2];
  int b_row0;
  int b_rows;    // rows of B = MMA N
  int k0;        // first contraction element
  int kstages;
  int klast;     // contraction elements of the last stage
  int out_row0;
  int out_col0;
  long long sfa_atom[2];  // atom index of stage 0 for each A tile
  long long sfb_atom;     // atom index of stage 0 for B
};

struct MetaCache {
  const int4* blocks;   // grouped-M: s_blocks[b] for b < ncache
  int ncache = kCacheBlocks;
  const int* poff;      // grouped-K: poffsets[0..E]
  const int* bstart;    // grouped-K: bstart[0..E]
};

// STEP: weight rows per grouped-M output tile: 128, or 256 when the two A
// tiles of an NA = 2 store tile are adjacent 128-row blocks (the SwiGLU
// forward's second A tile is the up half, F rows on); over row-block pairs,
// 128 (store) or 64 (SwiGLU forward: 64 features, their gate and up rows).
//
// Grouped-M tiles run routing block by routing block, all output slices of
// a block together: the resident CTAs then cover a few blocks at a time,
// each block's activation rows come from DRAM once and are shared in L2 by
// the CTAs of its slices, and the blocks of one expert (adjacent in block
// order) still read the same weight slices at about the same time.  Slice
// by slice instead, the weight stream evicts every activation bundle larger
// than a few tens of MB from L2 before the next slice comes back to it.
//
// A CTA's tiles are tile0, tile0 + step, ...: the walk keeps their
// coordinates (grouped-M: block m and slice n, tile = m * n_tiles + n;
// grouped-K: expert e, m, n, tile = (e * m_tiles + m) * n_tiles + n) and
// advances them by the step's own coordinates with carries, so no role
// divides per tile.  (Weight-gradient tiles are mostly one stage deep, and
// two integer divisions per tile sat on the MMA thread's serial path.)
template <int MODE>
struct TileWalk {
  int tile, n, m, e;
  // the walk's step comes from p.walk (parameter space, no registers)
  __device__ __forceinline__ void start(const GemmParams& p, int tile0) {
    tile = tile0;
    n = tile0 % p.n_tiles;
    const int q = tile0 / p.n_tiles;
    m = MODE != kGroupedK ? q : q % p.m_tiles;
    e = MODE != kGroupedK ? 0 : q / p.m_tiles;
  }
  __device__ __forceinline__ void advance(const GemmParams& p) {
    tile += p.walk[0];
    n += p.walk[1];
    const int c = n >= p.n_tiles;
    n -= c ? p.n_tiles : 0;
    m += p.walk[2] + c;
    if (MODE == kGroupedK) {
      const int c2 = m >= p.m_tiles;
      m -= c2 ? p.m_tiles : 0;
      e += p.walk[3] + c2;
    }
  }
};

template <int MODE, int BK, int STEP>
__device__ __forceinline__ Tile decode_tile(const GemmParams& p, const TileWalk<MODE>& w, const MetaCache& mc) {
  Tile t;
  if (MODE == kGroupedM) {
    const int b = w.m, n = w.n;
    const int4 blk = (b < mc.ncache) ? mc.blocks[b] : p.blocks[b];
    t.e = blk.x;
    t.blk = b;
    t.a_row[0] = blk.x * p.a_rows_per_expert + n * STEP;
    t.a_row[1] = t.a_row[0] + (STEP == 256 ? 128 : p.a_up_offset);
    t.b_row0 = blk.y;
    t.b_rows = blk.z;
    t.k0 = 0;
    t.kstages = p.K / BK;
    t.klast = BK;
    t.out_row0 = blk.y;
    t.out_col0 = n * STEP;
    t.sfa_atom[0] = static_cast<long long>(t.a_row[0] >> 7) * p.sfa_ts;
    t.sfa_atom[1] = static_cast<long long>(t.a_row[1] >> 7) * p.sfa_ts;
    t.sfb_atom = static_cast<long long>(b) * p.sfb_ts;
  } else if (MODE == kGroupedMP || MODE == kGroupedMC) {
    // pair m: word 3 of blocks[m] = (first block << 1) | second present;
    // the first block of a two-block pair is a full 128 rows
    const int m = w.m, n = w.n;
    const int desc = ((m < mc.ncache) ? mc.blocks[m] : p.blocks[m]).w;
    const int fb = desc >> 1;
    const int4 b0 = (fb < mc.ncache) ? mc.blocks[fb] : p.blocks[fb];
    t.e = b0.x;
    t.blk = fb;
    t.a_row[0] = b0.x * p.a_rows_per_expert + n * STEP;
    t.a_row[1] = t.a_row[0] + (STEP == 64 ? p.a_up_offset : 0);
    t.b_row0 = b0.y;
    t.b_rows = (desc & 1) ? 128 + ((fb + 1 < mc.ncache) ? mc.blocks[fb + 1] : p.blocks[fb + 1]).z : b0.z;
    t.k0 = 0;
    t.kstages = p.K / BK;
    t.klast = BK;
    t.out_row0 = b0.y;
    t.out_col0 = n * STEP;
    t.sfa_atom[0] = static_cast<long long>(t.a_row[0] >> 7) * p.sfa_ts;
    t.sfa_atom[1] = static_cast<long long>(t.a_row[1] >> 7) * p.sfa_ts;
    t.sfb_atom = static_cast<long long>(fb) * p.sfb_ts;
  } else {
    const int e = w.e, m = w.m, n = w.n;
    const int k0 = mc.poff[e], klen = mc.poff[e + 1] - k0;
    t.e = e;
    t.blk = 0;
    t.a_row[0] = m * 128;
    t.a_row[1] = 0;
    t.b_row0 = n * 128;
    t.b_rows = 128;
    t.k0 = k0;
    t.kstages = (klen + BK - 1) / BK;
    t.klast = klen - (t.kstages - 1) * BK;
    t.out_row0 = m * 128;
    t.out_col0 = n * 128;
    const int b0 = mc.bstart[e];
    t.sfa_atom[0] = static_cast<long long>(m) * p.sfa_ts + b0;
    t.sfa_atom[1] = 0;
    t.sfb_atom = static_cast<long long>(n) * p.sfb_ts + b0;
  }
  return t;
}

// Width in bytes of the K-major rows a stage loads: 128 (a full stage), or
// for the last stage of a weight-gradient tile only as much as it holds
// (32 or 64 bytes when that is enough), so short experts do not stream
// unused columns through TMA and shared memory.
template <int MODE, int BK, int ESZ>
__device__ __forceinline__ int stage_row_bytes(const Tile& t, int ks) {
  if (MODE != kGroupedK || ks != t.kstages - 1) return 128;
  const int b = t.klast * ESZ;
  return b <= 32 ? 32 : (b <= 64 ? 64 : 128);
}

// A final bounded wait that ignores the abort flag (used only to drain work
// already in flight before the CTA releases its resources).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitTimeoutCycles / 8) return;
  }
}

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

// Row bundle of one 32-feature block held across the warp's lanes (MXFP8:
// the block's amax is a warp reduction; the scale goes to the row-bundle
// atom of routing block `blk`, row `prow` within it).
template <bool MX>
__device__ __forceinline__ void store_row_val(const GemmParams& p, void* out, long long pitch, long long row,
                                              int col, float v, int lane, int blk, int prow) {
  if (!MX) {
    static_cast<__nv_bfloat16*>(out)[row * pitch + col] = __float2bfloat16_rn(v);
  } else {
    const float amax = warp_max_nonneg(fabsf(v));
    const int e = mx_shared_exp(amax);
    const uint32_t code = cvt_e4m3x2(v * exp2_int(-e), 0.0f) & 0xFFu;
    static_cast<uint8_t*>(out)[row * pitch + col] = static_cast<uint8_t>(code);
    if (lane == 0) {
      const int kb = col >> 5;
      p.out0_sf[(static_cast<long long>(blk) * p.out0_sf_kg + (kb >> 2)) * kAtom + sf_atom_byte(prow, kb & 3)] =
          static_cast<uint8_t>(e + 127);
    }
  }
}

// Column bundle: 32 rows of one feature in one thread's registers, written
// contiguously to outT[feat][row0 ..]; MXFP8 scale to the column-bundle atom
// (feature tile feat/128, routing block blk, 32-row group l).
template <bool MX>
__device__ __forceinline__ void store_col32(const GemmParams& p, long long feat, long long row0, int blk, int l,
                                            const float (&v)[32]) {
  if (!MX) {
    uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out1) + feat * p.out1_pitch + row0);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                        pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
  } else {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int e = mx_shared_exp(amax);
    const float inv = exp2_int(-e);
    uint32_t w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      w[q] = cvt_e4m3x2(v[4 * q] * inv, v[4 * q + 1] * inv) | (cvt_e4m3x2(v[4 * q + 2] * inv, v[4 * q + 3] * inv) << 16);
    uint4* o = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out1) + feat * p.out1_pitch + row0);
    o[0] = make_uint4(w[0], w[1], w[2], w[3]);
    o[1] = make_uint4(w[4], w[5], w[6], w[7]);
    p.out1_sf[((feat >> 7) * p.b_cap + blk) * kAtom + sf_atom_byte(static_cast<int>(feat & 127), l)] =
        static_cast<uint8_t>(e + 127);
  }
}

// ------------------------------------------------------------- epilogues
// Each takes the warp's chunk index `h` (0 or 1) and drains the 32-column
// chunks c0 = 32h and 32h + 64.  The store and SwiGLU-forward epilogues hand
// the accumulator back (`tempty`) as soon as their last TMEM read has
// landed, before the stores, so the next tile's MMAs overlap the store work
// (with two A tiles per stage there is a single 256-column accumulator).

// This warp is done reading the accumulator.
__device__ __forceinline__ void release_acc(uint64_t* tempty, int lane) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(tempty);
}

// h3 / input-gradient rows: out[row][feature] = bf16(acc).
// With NA = 2 the two accumulators hold features out_col0 + [0, 128) and
// out_col0 + [128, 256).  NC: chunks per warp (2: up to 128 token columns,
// 4: a row-block pair's 256).  Every chunk is read from TMEM first, rounded
// to BF16 pairs at once (the stored value), and the accumulator handed back
// before the first store.
template <int NA, int NC = 2>
__device__ __forceinline__ void epi_store(const GemmParams& p, const Tile& t, uint32_t tbase, int lrow, int lane,
                                          int h, uint64_t* tempty) {
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out0);
  uint32_t pk[NA][NC][16];
#pragma unroll
  for (int ci = 0; ci < NC; ++ci) {
    const int c0 = 32 * h + 64 * ci;
    if (c0 < t.b_rows) {
      uint32_t v[NA][32];   // both accumulators' chunk, one wait
#pragma unroll
      for (int j = 0; j < NA; ++j) tmem_ld32(tbase + j * 128 + c0, v[j]);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < NA; ++j)
#pragma unroll
        for (int q = 0; q < 16; ++q) pk[j][ci][q] = pack_bf16x2(u2f(v[j][2 * q]), u2f(v[j][2 * q + 1]));
    }
  }
  release_acc(tempty, lane);
#pragma unroll
  for (int j = 0; j < NA; ++j)
#pragma unroll
    for (int ci = 0; ci < NC; ++ci) {
      const int c0 = 32 * h + 64 * ci;
      if (c0 < t.b_rows) {
        __nv_bfloat16* o = out + static_cast<long long>(t.out_row0 + c0) * p.out0_pitch + t.out_col0 + j * 128 + lrow;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t w = pk[j][ci][i >> 1];
          o[static_cast<long long>(i) * p.out0_pitch] =
              __ushort_as_bfloat16(static_cast<unsigned short>((i & 1) ? (w >> 16) : (w & 0xFFFFu)));
        }
      }
    }
}

// One 32-token chunk of feature f: gu[i] = (g, u) of token row row0 + i as
// a BF16 pair; the rows lie in routing block blk from its row prow0 on.
template <bool MX>
__device__ __forceinline__ void swiglu_fwd_chunk(const GemmParams& p, long long row0, int f, int blk, int prow0,
                                                 const uint32_t (&gu)[32], int lane) {
  float hv[32];
  const float L = p.swiglu_limit;
  int cg = 0, cu = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const long long row = row0 + i;
    const uint32_t w = gu[i];
    if (p.save_h1) {
      p.h1[row * p.h1_pitch + f] = __ushort_as_bfloat16(static_cast<unsigned short>(w & 0xFFFFu));
      p.h1[row * p.h1_pitch + p.F + f] = __ushort_as_bfloat16(static_cast<unsigned short>(w >> 16));
    }
    float g = bf16_lo(w), u = bf16_hi(w);
    if (L > 0.0f) {
      cg += g > L;
      cu += fabsf(u) > L;
      g = fminf(g, L);
      u = fminf(fmaxf(u, -L), L);
    }
    hv[i] = silu_f(g) * u;
  }
  if (L > 0.0f && p.clip != nullptr) {
    cg = __reduce_add_sync(0xFFFFFFFFu, cg);
    cu = __reduce_add_sync(0xFFFFFFFFu, cu);
    if (lane == 0) {
      if (cg) atomicAdd(&p.clip[0], static_cast<unsigned long long>(cg));
      if (cu) atomicAdd(&p.clip[1], static_cast<unsigned long long>(cu));
    }
  }
#pragma unroll
  for (int i = 0; i < 32; ++i)
    store_row_val<MX>(p, p.out0, p.out0_pitch, row0 + i, f, hv[i], lane, blk, prow0 + i);
  if (p.want_col) store_col32<MX>(p, f, row0, blk, prow0 >> 5, hv);
}

// Fused SwiGLU forward: g, u from the two accumulators, rounded to BF16
// (the stored h1), h2 = SiLU(g) * u in FP32, then the h2 row bundle (W2's
// operand) and, for training, the h2 column bundle (W2 WGRAD's operand).
// Both chunks are read from TMEM first, as BF16 (g, u) pairs (the stored
// h1 and the SwiGLU's inputs), and the accumulator handed back before any
// store.  With a limit L > 0 (clamped SwiGLU, "Meta Dist-MoE: Open-Source
// Fused MoE Kernels for Blackwell", "Supported modes") g is clamped to <= L
// and u to [-L, L] first; the warp counts the values it clamps (clip
// statistics) and adds them to p.clip once per chunk.  h1 keeps the
// unclamped values, which the backward needs for its masks.
template <bool MX>
__device__ __forceinline__ void epi_swiglu_fwd(const GemmParams& p, const Tile& t, uint32_t tbase, int lrow,
                                               int lane, int h, uint64_t* tempty) {
  const int f = t.out_col0 + lrow;
  uint32_t gu[2][32];
#pragma unroll
  for (int ci = 0; ci < 2; ++ci) {
    const int c0 = 32 * h + 64 * ci;
    if (c0 < t.b_rows) {
      uint32_t vg[32], vu[32];
      tmem_ld32(tbase + c0, vg);
      tmem_ld32(tbase + 128 + c0, vu);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) gu[ci][i] = pack_bf16x2(u2f(vg[i]), u2f(vu[i]));
    }
  }
  release_acc(tempty, lane);
#pragma unroll
  for (int ci = 0; ci < 2; ++ci) {
    const int c0 = 32 * h + 64 * ci;
    if (c0 < t.b_rows) swiglu_fwd_chunk<MX>(p, t.out_row0 + c0, f, t.blk, c0, gu[ci], lane);
  }
}

// Fused SwiGLU forward over a row-block pair.  The A tile is 64 gate rows
// and then the 64 up rows of the same features, so TMEM lanes 0..63 hold g
// and lanes 64..127 u: the warp of lane quadrant q < 2 and the warp of
// quadrant q + 2 with the same chunk set h hold g and u of the same 32
// features (feature out_col0 + 32 q + lane).  Of their four 32-token chunks
// (columns 32 h + 64 ci), the gate warp finishes ci = 0 and 2 and the up
// warp ci = 1 and 3; each hands the other its BF16 values (the stored h1) of
// the partner's chunks through `xbuf`, 16 KB per round, two rounds.  Every
// epilogue warp passes the same named barriers; if any warp's accumulator
// wait gave up (`ok` false), all leave together and it returns false.
template <bool MX>
__device__ __forceinline__ bool epi_swiglu_fwd_pair(const GemmParams& p, const Tile& t, uint32_t tbase, int q,
                                                    int lane, int h, bool ok, uint64_t* tempty, uint8_t* xbuf,
                                                    volatile int* abort_flag, int bar_id, int bar_threads) {
  const int up = q >> 1, qg = q & 1;
  const int f = t.out_col0 + 32 * qg + lane;
  uint4* mine = reinterpret_cast<uint4*>(xbuf + (((qg * 2 + h) * 2 + up) << 11));
  const uint4* theirs = reinterpret_cast<const uint4*>(xbuf + (((qg * 2 + h) * 2 + (up ^ 1)) << 11));
  if (!ok && lane == 0) *abort_flag = 1;
  named_bar_sync(bar_id, bar_threads);
  if (*abort_flag) return false;
  uint32_t own[2][16], oth[16], par[2][16];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int co = 32 * h + 64 * (2 * k + up), cx = 32 * h + 64 * (2 * k + (up ^ 1));
    uint32_t vo[32], vx[32];
    if (co < t.b_rows) tmem_ld32(tbase + co, vo);
    if (cx < t.b_rows) tmem_ld32(tbase + cx, vx);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      own[k][i] = pack_bf16x2(u2f(vo[2 * i]), u2f(vo[2 * i + 1]));
      oth[i] = pack_bf16x2(u2f(vx[2 * i]), u2f(vx[2 * i + 1]));
    }
    if (k == 0 && cx < t.b_rows) {
#pragma unroll
      for (int j = 0; j < 4; ++j) mine[j * 32 + lane] = make_uint4(oth[4 * j], oth[4 * j + 1], oth[4 * j + 2], oth[4 * j + 3]);
    }
  }
  release_acc(tempty, lane);
  const int co0 = 32 * h + 64 * up, co1 = co0 + 128, cx1 = 32 * h + 64 * (2 + (up ^ 1));
  named_bar_sync(bar_id, bar_threads);   // round 0 written
  if (co0 < t.b_rows) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 w = theirs[j * 32 + lane];
      par[0][4 * j] = w.x;
      par[0][4 * j + 1] = w.y;
      par[0][4 * j + 2] = w.z;
      par[0][4 * j + 3] = w.w;
    }
  }
  named_bar_sync(bar_id, bar_threads);   // round 0 read
  if (cx1 < t.b_rows) {
#pragma unroll
    for (int j = 0; j < 4; ++j) mine[j * 32 + lane] = make_uint4(oth[4 * j], oth[4 * j + 1], oth[4 * j + 2], oth[4 * j + 3]);
  }
  named_bar_sync(bar_id, bar_threads);   // round 1 written
  if (co1 < t.b_rows) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 w = theirs[j * 32 + lane];
      par[1][4 * j] = w.x;
      par[1][4 * j + 1] = w.y;
      par[1][4 * j + 2] = w.z;
      par[1][4 * j + 3] = w.w;
    }
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int co = k ? co1 : co0;
    if (co >= t.b_rows) continue;
    uint32_t gu[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t g2 = up ? par[k][i] : own[k][i], u2 = up ? own[k][i] : par[k][i];
      gu[2 * i] = __byte_perm(g2, u2, 0x5410);       // (g, u) of token 2i
      gu[2 * i + 1] = __byte_perm(g2, u2, 0x7632);   // of token 2i + 1
    }
    swiglu_fwd_chunk<MX>(p, t.out_row0 + co, f, t.blk + (co >> 7), co & 127, gu, lane);
  }
  return true;
}

// Fused SwiGLU backward: dh2 from the accumulator (W2 DGRAD), g and u from
// the saved BF16 h1, dg = dh2 u SiLU'(g), du = dh2 SiLU(g), written as the
// dh1 row bundle (W13 DGRAD's operand) and column bundle (W13 WGRAD's).
// With a clamp limit L, g and u are clamped first and dg (du) is zero where
// g > L (|u| > L).
// h1 does not depend on the MMA, so the caller issues the loads of the
// warp's first chunk before it waits for the accumulator.
__device__ __forceinline__ void load_h1_chunk(const GemmParams& p, const Tile& t, int f, int c0,
                                              uint32_t (&hp)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    hp[i] = 0;
    if (c0 + i < t.b_rows) {
      const long long row = t.out_row0 + c0 + i;
      const uint32_t g = __bfloat16_as_ushort(p.h1[row * p.h1_pitch + f]);
      const uint32_t u = __bfloat16_as_ushort(p.h1[row * p.h1_pitch + p.F + f]);
      hp[i] = g | (u << 16);
    }
  }
}

template <bool MX>
__device__ __forceinline__ void epi_swiglu_bwd(const GemmParams& p, const Tile& t, uint32_t tbase, int lrow,
                                               int lane, int h, uint32_t (&hp)[32]) {
  const int f = t.out_col0 + lrow;
  for (int c0 = 32 * h; c0 < t.b_rows; c0 += 64) {
    if (c0 != 32 * h) load_h1_chunk(p, t, f, c0, hp);   // the first chunk was prefetched
    uint32_t v[32];
    tmem_ld32(tbase + c0, v);
    tmem_ld_wait();
    float dg[32], du[32];
    const float L = p.swiglu_limit;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float g = bf16_lo(hp[i]);
      float u = bf16_hi(hp[i]);
      const float dh2 = u2f(v[i]);
      float mg = 1.0f, mu = 1.0f;   // clamped SwiGLU: gradient only inside the clamp range
      if (L > 0.0f) {
        mg = g <= L ? 1.0f : 0.0f;
        mu = fabsf(u) <= L ? 1.0f : 0.0f;
        g = fminf(g, L);
        u = fminf(fmaxf(u, -L), L);
      }
      const float s = sigmoid_f(g);
      dg[i] = dh2 * u * (s * (1.0f + g * (1.0f - s))) * mg;
      du[i] = dh2 * (g * s) * mu;
    }
    // over a row-block pair, rows 128.. of the tile are the second block's
    const int blk = t.blk + (c0 >> 7), prow = c0 & 127;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const long long row = t.out_row0 + c0 + i;
      store_row_val<MX>(p, p.out0, p.out0_pitch, row, f, dg[i], lane, blk, prow + i);
      store_row_val<MX>(p, p.out0, p.out0_pitch, row, p.F + f, du[i], lane, blk, prow + i);
    }
    store_col32<MX>(p, f, t.out_row0 + c0, blk, prow >> 5, dg);
    store_col32<MX>(p, p.F + f, t.out_row0 + c0, blk, prow >> 5, du);
  }
}

// Weight gradient with plain stores: dW[e][m][n0 ..], FP32 or accumulate.
// An expert without rows gets zeros, or is left as is when adding.  A lane
// holds one row of each 32 x 32 chunk it drains; the warp turns the chunk
// around in its own 4 KB of the group's staging buffer (float4 slots
// XOR-swizzled by row: conflict-free writes and reads) so that each global
// load and store covers 4 rows x 32 consecutive columns instead of 32 rows.
__device__ __forceinline__ void epi_wgrad_direct(const GemmParams& p, const Tile& t, uint32_t tbase, int q, int lane,
                                                 int h, int step, float* ws) {
  if (t.kstages == 0 && p.dw_accum) return;
  const long long M = static_cast<long long>(p.m_tiles) * 128;
  const long long row0 = static_cast<long long>(t.e) * M + t.out_row0 + q * 32;   // the warp's first row
  const int rr = lane >> 3, j = lane & 7;   // read-back: rows rr, rr + 4, ...; float4 slot j of each
  for (int c0 = 32 * h; c0 < 128; c0 += step) {
    uint32_t r[32];   // FP32 bits of the chunk's row
    if (t.kstages > 0) {
      tmem_ld32(tbase + c0, r);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = 0u;
    }
#pragma unroll
    for (int s4 = 0; s4 < 8; ++s4)
      *reinterpret_cast<uint4*>(ws + lane * 32 + ((s4 ^ (lane & 7)) << 2)) =
          make_uint4(r[4 * s4], r[4 * s4 + 1], r[4 * s4 + 2], r[4 * s4 + 3]);
    __syncwarp();
#pragma unroll 2
    for (int it = 0; it < 8; ++it) {
      const int r = 4 * it + rr;
      float4 a = *reinterpret_cast<const float4*>(ws + r * 32 + ((j ^ (r & 7)) << 2));
      const long long off = (row0 + r) * p.out0_pitch + t.out_col0 + c0 + 4 * j;
      if (p.dw_fp32) {
        float4* o = reinterpret_cast<float4*>(static_cast<float*>(p.out0) + off);
        if (p.dw_accum) {
          const float4 y = *o;
          a.x += y.x;
          a.y += y.y;
          a.z += y.z;
          a.w += y.w;
        }
        *o = a;
      } else {
        uint2* o = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out0) + off);
        if (p.dw_accum) {
          const uint2 y = *o;
          a.x += bf16_lo(y.x);
          a.y += bf16_hi(y.x);
          a.z += bf16_lo(y.y);
          a.w += bf16_hi(y.y);
        }
        *o = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
      }
    }
    __syncwarp();   // every lane has read the chunk before the next one overwrites it
  }
}

// Weight gradient (BF16, overwrite) through shared memory: the 128 x 128
// tile is written into a 32 KB staging buffer as two 128-row x 128-byte
// boxes in the 128-byte swizzle (16-byte chunk j of row m at chunk
// j ^ (m % 8), so 8 consecutive rows hit 8 different bank groups), then one
// thread stores both boxes with TMA.  `r` holds the 32 columns from c0 of
// row lrow, already loaded from TMEM.
__device__ __forceinline__ void stage_chunk(const uint32_t (&r)[32], bool zero, int c0, int lrow, uint8_t* stg) {
  uint8_t* box = stg + (c0 >> 6) * 16384 + lrow * 128;
  const int j0 = (c0 & 63) >> 3;  // first 16-byte chunk of these 32 columns
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int phys = (j0 + q) ^ (lrow & 7);
    uint4 w = make_uint4(0, 0, 0, 0);
    if (!zero)
      w = make_uint4(pack_bf16x2(u2f(r[8 * q + 0]), u2f(r[8 * q + 1])), pack_bf16x2(u2f(r[8 * q + 2]), u2f(r[8 * q + 3])),
                     pack_bf16x2(u2f(r[8 * q + 4]), u2f(r[8 * q + 5])), pack_bf16x2(u2f(r[8 * q + 6]), u2f(r[8 * q + 7])));
    *reinterpret_cast<uint4*>(box + phys * 16) = w;
  }
}

// Weight gradient in FP32 through shared memory: 32 FP32 columns (c0 ..
// c0 + 31 of the half tile being staged) of row lrow into one 128-row x
// 128-byte box of the 32 KB staging buffer (box = which 32 columns of the
// half), in the same 128-byte swizzle.
__device__ __forceinline__ void stage_chunk_f32(const uint32_t (&r)[32], bool zero, int box, int lrow, uint8_t* stg) {
  uint8_t* row = stg + box * 16384 + lrow * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 w = zero ? make_uint4(0, 0, 0, 0) : make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
    *reinterpret_cast<uint4*>(row + ((j ^ (lrow & 7)) << 4)) = w;
  }
}

// ------------------------------------------------------------------ kernel

template <bool MX, int NA, int MODE>
struct Cfg {
  static constexpr bool WGRAD = MODE == kGroupedK;
  // over row-block pairs: one A tile, a B operand of up to 256 rows (two
  // 128-row boxes), scale atoms of two A halves (gate, up) and two B blocks
  static constexpr bool PAIR = MODE == kGroupedMP || MODE == kGroupedMC;
  // over row-block pairs on a CTA pair: this CTA's B is one block (128 rows)
  // of the pair; both B atoms, as every SM's MMA reads the scales of all 256.
  // A stage holds two K-chunks (K = 256): the operands come in one box each
  // (two 16 KB chunk tiles) and the scale atoms of both chunks in one copy
  // per operand, so each SM fills three 68 KB stages with five copies per
  // stage (large stages and few copies are what keeps the L2-to-shared-
  // memory stream near 24 TB/s for the whole GPU; 32 KB stages of two boxes
  // and three small copies reach about 10).
  static constexpr bool CG2 = MODE == kGroupedMC;
  static_assert(!PAIR || NA == 1, "one A tile per stage over row-block pairs");
  static constexpr int KCH = CG2 ? 2 : 1;                  // 128-element K-chunks per stage
  static constexpr int SF_BYTES = MX ? (PAIR ? 4 * KCH : NA + 1) * kAtom : 0;
  // Scale-atom groups (MXFP8, grouped-M, one A tile): the atoms of GS
  // consecutive stages of a tile are consecutive in memory for the weight
  // and for the row block, so they come in two copies per group into a
  // ring of their own instead of two per stage (each TMA copy has a fixed
  // cost well above its 512 bytes; this GEMM streams only 16 KB of weights
  // per stage).
  static constexpr bool SFG = MX && MODE == kGroupedM && NA == 1;
  static constexpr int GS = 4, SFR = 2;
  static constexpr int GROUP_BYTES = GS * (NA + 1) * kAtom;
  static constexpr int SFG_BYTES = SFG ? SFR * GROUP_BYTES : 0;
  static constexpr int A_BYTES = NA * KCH * kABytes;
  static constexpr int B_BYTES = (PAIR && !CG2) ? 2 * kBBytes : KCH * kBBytes;
  static constexpr int SF_OFF = A_BYTES + B_BYTES;           // a stage's scale atoms
  static constexpr int STAGE = ((SF_OFF + (SFG ? 0 : SF_BYTES)) + 1023) / 1024 * 1024;
  static constexpr int S = CG2 ? 3 : (WGRAD ? 4 : ((NA == 2 || PAIR) ? 4 : 6));  // pipeline stages
  static constexpr int STAGING = WGRAD ? 2 * 32768 : 0;    // weight-gradient store buffers
  // accumulator buffers: two, except with two MXFP8 A tiles or a 256-wide
  // MXFP8 pair tile (2 x 256 columns leave no room in TMEM's 512 for the
  // stages' scale columns)
  static constexpr int ACC_BUFS = PAIR ? (MX ? 1 : 2) : ((NA == 1 || !MX) ? 2 : 1);
  static constexpr int ACC_COLS = PAIR ? 256 : NA * 128;
  static constexpr int SF_COLS = PAIR ? 12 * KCH : (NA + 1) * 4;  // scale columns per stage (B: 8 over pairs)
  // the pair SwiGLU epilogue's exchange buffer; a smaller metadata cache
  static constexpr int EXCH = PAIR ? 16384 : 0;
  static constexpr int CACHE = CG2 ? 4096 : (PAIR ? 8192 : kCacheBytes);
  // mbarriers, the TMEM address and the abort flags (CTA pairs: also each
  // stage's "both CTAs' operands are ready" and the other CTA's accumulator
  // release)
  static constexpr int BARS = CG2 ? 512 : 256;
  static constexpr uint32_t SF_COL0 = ACC_BUFS * ACC_COLS;
  static constexpr int BK = (MX ? 128 : 64) * KCH;         // contraction elements per stage
  static constexpr int KMMA = MX ? 32 : 16;                // contraction elements per MMA
  static constexpr int MMAS = BK / KMMA;
  // epilogue warps: 8 (two per TMEM lane quadrant, alternate 32-column
  // chunks).  The weight-gradient GEMM, whose per-tile work is almost all
  // epilogue, has two such groups of 8 that take alternate tiles (one
  // accumulator buffer, staging buffer and named barrier each), so the
  // TMEM-load -> stage -> store chains of two tiles overlap.
  static constexpr int EPI_GROUPS = WGRAD ? 2 : 1;
  static constexpr int EPI_WARPS = 8 * EPI_GROUPS;
  static constexpr int EPI_THREADS = EPI_WARPS * 32;
  static constexpr int GROUP_THREADS = EPI_THREADS / EPI_GROUPS;
  static_assert(!WGRAD || (NA == 1 && ACC_BUFS == EPI_GROUPS), "one accumulator buffer per epilogue group");
  // MXFP8: one more warp copies each stage's scale atoms to TMEM, so the
  // MMA thread issues nothing but MMAs and commits (CTA pairs, BF16 too: it
  // reports each stage to rank 0)
  static constexpr int SF_WARPS = (MX || CG2) ? 1 : 0;
  static constexpr int THREADS = 64 + EPI_THREADS + 32 * SF_WARPS;
  static constexpr int SMEM = 1024 + S * STAGE + STAGING + SFG_BYTES + EXCH + BARS + CACHE;
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static_assert(ACC_BUFS * ACC_COLS + S * (MX ? SF_COLS : 0) <= 512, "tensor memory columns");
};

}  // namespace

}  // namespace moe
