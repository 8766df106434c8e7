// Single-launch inference forward (MXFP8): routing, gather, W13 + SwiGLU,
// W2 and combine in one persistent grid.
//
// "Dist-MoE: Speed-of-light distributed Mixture-of-Experts kernels", section
// 05, "Kernel Pipelines: Staged and Mega": the staged forward runs ordered
// launches; the Mega forward joins W13 and W2 in one grid whose resident
// CTAs repeat work records on fixed warp roles (the same TMA, MMA and
// epilogue roles serve W13 and W2) and coordinate through readiness
// counters in global memory.  Here the grid also takes the routing, the
// gather and the combine, so a decode-sized step is one launch.  "Mixture of Experts: How Routing Becomes GPU Computation",
// section 6: with few tokens, W13 has too few output tiles to fill the GPU;
// the CTAs that hold W2 tiles ask L2 for their first weight stages while
// the W13 tiles they depend on are still running, and every producer asks
// L2 for the weight stages a few ahead of the ones it loads.
//
// Work records, numbered once the routing is known (nblk row blocks):
//   [0, nblk gp)                   gather block b, column part p (x rows -> MXFP8 row bundle)
//   [.., + nblk n13)               W13 + SwiGLU tile (b, n), block-major
//   [.., + nblk n2)                W2 tile (b, n), block-major
//   [.., + 4 T)                    combine: a quarter of token t's columns
// CTA i takes records i, i + grid, ... in increasing order, and every role
// of a CTA walks that sequence in order.  A record waits only for records
// numbered below it: a W13 tile for its block's gather, a W2 tile for its
// block's n13 W13 tiles, a combine for every W2 tile.  The lowest unfinished
// record therefore never waits, and the grid (at most one CTA per SM,
// launched cooperatively, so all CTAs are resident) always progresses.
// Every wait is bounded: it gives up after a deadline, sets the timeout bit
// and the CTA's abort flag, and the CTA leaves.
//
// The results equal the staged launches' bit for bit: the same routing,
// the same row-bundle codes, the same GEMM stages and MMA order, the same
// epilogues, the same fixed-order FP32 combine.
//
// Every CTA computes the routing's row blocks (its work records) from the
// IDs itself, and a gather record ranks its block's routes from the IDs, so
// no record waits for the routing arrays; the last CTA writes those arrays
// (the routing kernel's layout), which only the combine reads.
//
// Counters (ints in the context's scratch, zero between launches):
//   [0] routing arrays published   [1] CTAs finished   [2] W2 tiles finished
//   [3 + b]                 gather of block b finished
//   [3 + b_cap + b]         W13 tiles of block b finished
// The last CTA to finish returns them all to zero for the next launch.
#include <algorithm>

#include "gemm_core.cuh"

namespace moe {

namespace {

using CF = Cfg<true, 2, kGroupedM>;
constexpr int kFusedThreads = CF::THREADS;     // producer, MMA (and scale copies), 8 epilogue warps, one idle warp
constexpr int kEpiThreads = CF::EPI_THREADS;
constexpr int kFusedSmem = CF::SMEM + kBlockRows * 4;   // + a gather record's routes
constexpr int kPrefetch = 8;   // weight stages asked of L2 ahead of their loads
constexpr int kCombineParts = 4;   // combine records per token (D % (8 kCombineParts) == 0)

// Gather records per row block: column parts of D / gp columns, a multiple
// of 128 (whole scale atoms), so one block's gather spreads over gp CTAs.
__host__ __device__ __forceinline__ int gather_parts(int D) {
  const int atoms = D / 128;
  return atoms % 8 == 0 ? 8 : (atoms % 4 == 0 ? 4 : (atoms % 2 == 0 ? 2 : 1));
}

struct Rec {
  int kind;   // 0 gather, 1 W13 tile, 2 W2 tile, 3 combine
  int b, n;   // block and slice (tiles), block and column part (gather), combine part (b)
};

__device__ __forceinline__ Rec record(int u, int nblk, int gp, int n13, int n2) {
  Rec r{};
  if (u < nblk * gp) {
    r.kind = 0;
    r.b = u / gp;
    r.n = u - r.b * gp;   // column part
    return r;
  }
  u -= nblk * gp;
  if (u < nblk * n13) {
    r.kind = 1;
    r.b = u / n13;
    r.n = u - r.b * n13;
    return r;
  }
  u -= nblk * n13;
  if (u < nblk * n2) {
    r.kind = 2;
    r.b = u / n2;
    r.n = u - r.b * n2;
    return r;
  }
  r.kind = 3;
  r.b = u - nblk * n2;
  return r;
}

__device__ __forceinline__ Tile tile_of(const FusedArgs& fa, const Rec& r, const MetaCache& mc) {
  TileWalk<kGroupedM> w;
  w.tile = 0;
  w.e = 0;
  w.m = r.b;
  w.n = r.n;
  return r.kind == 1 ? decode_tile<kGroupedM, CF::BK, 128>(fa.g13, w, mc)
                     : decode_tile<kGroupedM, CF::BK, 256>(fa.g2, w, mc);
}

// ------------------------------------------------------- local block list
// Every CTA, all threads: the row blocks of the routing, computed from the
// IDs into the CTA's block cache (the same blocks, in the same order, as the
// routing kernel's list; the fourth field holds the rank of the block's
// first row among its expert's routes), so no CTA waits for another to
// learn its work records.  `ws` is shared scratch of E ints.
__device__ void local_blocks(const FusedArgs& fa, int* ws, int4* cache, volatile int* s_nblk) {
  const int E = fa.E, TK = fa.T * fa.K;
  const int tid = threadIdx.x, lane = tid & 31;
  for (int e = tid; e < E; e += blockDim.x) ws[e] = 0;
  __syncthreads();
  for (int i = tid; i < TK; i += blockDim.x) {
    const int id = __ldg(fa.ids + i);
    if (id >= 0 && id < E) atomicAdd(&ws[id], 1);
  }
  __syncthreads();
  if (tid < 32) {
    int cp = 0, cb = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int c = e < E ? ws[e] : 0;
      const int pc = (c + kPad - 1) / kPad * kPad;
      const int nb = (pc + kBlockRows - 1) / kBlockRows;
      int ip = pc, ib = nb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int b = __shfl_up_sync(0xFFFFFFFFu, ip, o);
        const int d = __shfl_up_sync(0xFFFFFFFFu, ib, o);
        if (lane >= o) {
          ip += b;
          ib += d;
        }
      }
      const int ep = cp + ip - pc, eb = cb + ib - nb;
      for (int j = 0; j < nb; ++j)
        cache[eb + j] = make_int4(e, ep + j * kBlockRows, min(kBlockRows, pc - j * kBlockRows), j * kBlockRows);
      cp += __shfl_sync(0xFFFFFFFFu, ip, 31);
      cb += __shfl_sync(0xFFFFFFFFu, ib, 31);
    }
    if (lane == 0) *s_nblk = cb;
  }
  __syncthreads();
}

// ------------------------------------------------------------------ routing
// One CTA, all threads: the same arrays as the routing kernel (counts,
// exclusive prefixes plain and padded to 32 rows, stable expert-major
// permutation and inverse, row blocks, the routing copy of the scores).
// `ws` is shared scratch of 3 E + 2 ints.
__device__ void fused_route(const FusedArgs& fa, int* ws) {
  const RoutingPtrs& rp = fa.rp;
  const int T = fa.T, K = fa.K, E = fa.E, TK = T * K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* cnt = ws;           // [E]
  int* next = ws + E;      // [E]: next free row of each expert
  int* pstart = ws + 2 * E;  // [E]: first row of each expert
  int* tot = ws + 3 * E;   // [0] error bits
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  if (tid == 0) tot[0] = 0;
  __syncthreads();
  unsigned my_err = 0;
  for (int i = tid; i < TK; i += blockDim.x) {
    const int id = fa.ids[i];
    const float s = fa.scores[i];
    const bool act = id >= 0 && id < E;
    if (act) atomicAdd(&cnt[id], 1);
    else if (id != -1) my_err |= kErrBadId;
    else if (fa.debug && s != 0.0f) my_err |= kErrInactiveScore;
    rp.scores[i] = act ? s : 0.0f;
  }
  if (my_err) atomicOr(reinterpret_cast<unsigned*>(&tot[0]), my_err);
  __syncthreads();
  // exclusive prefixes over the experts, 32 at a time (warp 0)
  if (warp == 0) {
    int co = 0, cp = 0, cb = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int c = e < E ? cnt[e] : 0;
      const int pc = (c + kPad - 1) / kPad * kPad;
      const int nb = (pc + kBlockRows - 1) / kBlockRows;
      int io = c, ip = pc, ib = nb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xFFFFFFFFu, io, o);
        const int b = __shfl_up_sync(0xFFFFFFFFu, ip, o);
        const int d = __shfl_up_sync(0xFFFFFFFFu, ib, o);
        if (lane >= o) {
          io += a;
          ip += b;
          ib += d;
        }
      }
      if (e < E) {
        const int eo = co + io - c, ep = cp + ip - pc, eb = cb + ib - nb;
        rp.counts[e] = c;
        rp.offsets[e] = eo;
        rp.poffsets[e] = ep;
        rp.bstart[e] = eb;
        pstart[e] = ep;
        next[e] = ep;
        for (int j = 0; j < nb; ++j) {
          const int rows_b = min(kBlockRows, pc - j * kBlockRows);
          rp.blocks[eb + j] = make_int4(e, ep + j * kBlockRows, rows_b, 0);
          for (int g = 0; g < rows_b / kPad; ++g) rp.row_block[(ep + j * kBlockRows) / kPad + g] = eb + j;
        }
      }
      co += __shfl_sync(0xFFFFFFFFu, io, 31);
      cp += __shfl_sync(0xFFFFFFFFu, ip, 31);
      cb += __shfl_sync(0xFFFFFFFFu, ib, 31);
    }
    if (lane == 0) {
      rp.offsets[E] = co;
      rp.poffsets[E] = cp;
      rp.bstart[E] = cb;
      rp.hdr[0] = T;
      rp.hdr[1] = cb;
      rp.hdr[2] = cp;
      rp.hdr[3] = co;
    }
    // stable scatter, 32 routes at a time in flat order: a route's row is
    // its expert's next row plus the number of lower lanes with its expert
    for (int i0 = 0; i0 < TK; i0 += 32) {
      const int i = i0 + lane;
      const int id = i < TK ? fa.ids[i] : -1;
      const int e = (id >= 0 && id < E) ? id : -1;
      const unsigned grp = __match_any_sync(0xFFFFFFFFu, e);
      if (e >= 0) {
        const int row = next[e] + __popc(grp & ((1u << lane) - 1u));
        rp.perm[row] = i;
        rp.inv[i] = row;
      } else if (i < TK) {
        rp.inv[i] = -1;
      }
      __syncwarp();
      if (e >= 0 && lane == __ffs(grp) - 1) next[e] += __popc(grp);
      __syncwarp();
    }
  }
  __syncthreads();
  // pad rows gather nothing
  for (int j = tid; j < E * kPad; j += blockDim.x) {
    const int e = j / kPad, k = j - e * kPad;
    const int row = pstart[e] + cnt[e] + k;
    const int end = pstart[e] + (cnt[e] + kPad - 1) / kPad * kPad;
    if (row < end) rp.perm[row] = -1;
  }
  if (tid == 0 && tot[0]) atomicOr(fa.g13.err, static_cast<uint32_t>(tot[0]));
}

// ----------------------------------------------------------- gather block b
// The 8 epilogue warps: the columns [part D/gp, (part+1) D/gp) of the
// row bundle of the block's routed rows, exactly as the inference gather
// writes them (4 lanes per 32-value block, E8M0 scale into the block's
// atoms).  Work items are (row, 8-value chunk)
// pairs spread over all 256 threads, four at a time with every load in
// flight before the first is used, so a block with a single routed row
// (one-token decode) still has all its loads in flight at once.
__device__ void fused_gather(const FusedArgs& fa, int b, int part, int gp, const int4 blk, int gtid, int* s_route) {
  // the routes of this block's rows: expert blk.x's routes of rank blk.w ..
  // blk.w + blk.z - 1 in flat order (one warp ranks them with ballots);
  // rows past the expert's routes are pad rows (-1)
  if (gtid < kBlockRows) s_route[gtid] = -1;
  named_bar_sync(kEpiBarrier, kEpiThreads);
  if (gtid < 32) {
    const int TK = fa.T * fa.K;
    int run = 0;
    for (int i0 = 0; i0 < TK; i0 += 32) {
      const int i = i0 + gtid;
      const bool mine = i < TK && __ldg(fa.ids + i) == blk.x;
      const unsigned m = __ballot_sync(0xFFFFFFFFu, mine);
      const int rank = run + __popc(m & ((1u << gtid) - 1u)) - blk.w;
      if (mine && rank >= 0 && rank < blk.z) s_route[rank] = i;
      run += __popc(m);
    }
  }
  named_bar_sync(kEpiBarrier, kEpiThreads);
  const int D = fa.D, K = fa.K;
  // the block's routed rows come first (ranks in order); the rest are pad
  // rows, which this gather leaves as they are: an MMA output row depends
  // only on its own B row, so whatever (finite) codes a pad row holds reach
  // only pad rows of h1, h2 and h3, which the combine never reads
  int nreal = 0;
  for (int i = 0; i < blk.z; ++i) nreal += s_route[i] >= 0 ? 1 : 0;
  const long long atom_row = static_cast<long long>(b) * (D / 128);
  const int cols = D / gp, c0 = part * cols;   // this record's columns: whole scale atoms
  const int chunks = cols / 8;         // a multiple of 4: a 4-lane group never straddles two rows
  const int items = nreal * chunks;
  constexpr int kBatch = 4;
  for (int i0 = 0; i0 < items; i0 += kBatch * kEpiThreads) {
    uint4 ub[kBatch];
    int rr[kBatch], cc[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = i0 + j * kEpiThreads + gtid;
      const int rl = i / chunks;
      rr[j] = blk.y + rl;
      cc[j] = c0 + (i - rl * chunks) * 8;
      ub[j] = make_uint4(0, 0, 0, 0);
      if (i < items) {
        const int route = s_route[rr[j] - blk.y];
        if (route >= 0)
          ub[j] = __ldg(reinterpret_cast<const uint4*>(fa.x + static_cast<long long>(route / K) * D + cc[j]));
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = i0 + j * kEpiThreads + gtid;   // uniform per 4-lane group (items is a multiple of 4)
      const uint4 u = ub[j];
      float v[8] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y),
                    bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w)};
      float amax = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(v[k]));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
      const int e = mx_shared_exp(amax);
      const float inv = exp2_int(-e);
      uint2 qv;
      qv.x = cvt_e4m3x2(v[0] * inv, v[1] * inv) | (cvt_e4m3x2(v[2] * inv, v[3] * inv) << 16);
      qv.y = cvt_e4m3x2(v[4] * inv, v[5] * inv) | (cvt_e4m3x2(v[6] * inv, v[7] * inv) << 16);
      if (i < items) {
        *reinterpret_cast<uint2*>(fa.xrow + static_cast<long long>(rr[j]) * D + cc[j]) = qv;
        if ((gtid & 3) == 0) {
          const int kb = cc[j] >> 5;
          fa.xsf[(atom_row + (kb >> 2)) * 512 + sf_atom_byte(rr[j] - blk.y, kb & 3)] = static_cast<uint8_t>(e + 127);
        }
      }
    }
  }
}

// ------------------------------------------------------------ combine part
// Record q: token q / kCombineParts, the part q % kCombineParts of its D
// columns (a one-token step spreads over kCombineParts CTAs).
// out[t] = bf16((accumulate ? out[t] : 0) + sum_k s h3[inv]) in FP32, k in
// order: the combine kernel's arithmetic, with h3 read through L2 (other
// CTAs wrote it in this launch).  Up to 8 routes at a time: their rows,
// scores and h3 chunks are all in flight before the ordered FMAs.
__device__ void fused_combine(const FusedArgs& fa, int q, int gtid) {
  const int D = fa.D, K = fa.K;
  const int t = q / kCombineParts, part = q - t * kCombineParts;
  const int c_end = (part + 1) * (D / kCombineParts);
  __nv_bfloat16* orow = fa.out + static_cast<long long>(t) * D;
  const __nv_bfloat16* h3 = static_cast<const __nv_bfloat16*>(fa.g2.out0);
  for (int c = part * (D / kCombineParts) + gtid * 8; c < c_end; c += kEpiThreads * 8) {
    float acc[8];
    if (fa.accumulate) {
      const uint4 u = *reinterpret_cast<const uint4*>(orow + c);
      acc[0] = bf16_lo(u.x);
      acc[1] = bf16_hi(u.x);
      acc[2] = bf16_lo(u.y);
      acc[3] = bf16_hi(u.y);
      acc[4] = bf16_lo(u.z);
      acc[5] = bf16_hi(u.z);
      acc[6] = bf16_lo(u.w);
      acc[7] = bf16_hi(u.w);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    }
    for (int k0 = 0; k0 < K; k0 += 8) {
      int r[8];
      float sc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        r[j] = k0 + j < K ? __ldcg(fa.rp.inv + t * K + k0 + j) : -1;
        sc[j] = k0 + j < K ? __ldcg(fa.rp.scores + t * K + k0 + j) : 0.0f;
      }
      uint4 u[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        u[j] = make_uint4(0, 0, 0, 0);
        if (r[j] >= 0) u[j] = __ldcg(reinterpret_cast<const uint4*>(h3 + static_cast<long long>(r[j]) * D + c));
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (r[j] < 0) continue;
        const float s = sc[j];
        acc[0] = fmaf(s, bf16_lo(u[j].x), acc[0]);
        acc[1] = fmaf(s, bf16_hi(u[j].x), acc[1]);
        acc[2] = fmaf(s, bf16_lo(u[j].y), acc[2]);
        acc[3] = fmaf(s, bf16_hi(u[j].y), acc[3]);
        acc[4] = fmaf(s, bf16_lo(u[j].z), acc[4]);
        acc[5] = fmaf(s, bf16_hi(u[j].z), acc[5]);
        acc[6] = fmaf(s, bf16_lo(u[j].w), acc[6]);
        acc[7] = fmaf(s, bf16_hi(u[j].w), acc[7]);
      }
    }
    *reinterpret_cast<uint4*>(orow + c) = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                                     pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  }
}

__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_forward_kernel(const __grid_constant__ CUtensorMap a13, const __grid_constant__ CUtensorMap sf13,
                         const __grid_constant__ CUtensorMap bx32, const __grid_constant__ CUtensorMap bx128,
                         const __grid_constant__ CUtensorMap a2, const __grid_constant__ CUtensorMap sf2,
                         const __grid_constant__ CUtensorMap bh32, const __grid_constant__ CUtensorMap bh128,
                         const FusedArgs fa) {
  constexpr int S = CF::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * CF::STAGE);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_abort = abort_flag + 1;
  volatile int* s_nblk = abort_flag + 2;
  uint8_t* cache = smem + S * CF::STAGE + 256;
  int* sync = fa.sync;
  int* gather_done = sync + 3;
  int* w13_done = sync + 3 + fa.b_cap;
  uint32_t* err = fa.g13.err;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, CF::EPI_WARPS);
    mbar_init(drain, 1);
    *abort_flag = 0;
    *epi_abort = 0;
    *s_nblk = 0;
    mbar_fence_init();
    tma_prefetch(&a13);
    tma_prefetch(&sf13);
    tma_prefetch(&bx32);
    tma_prefetch(&bx128);
    tma_prefetch(&a2);
    tma_prefetch(&sf2);
    tma_prefetch(&bh32);
    tma_prefetch(&bh128);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- every CTA: the row blocks (its work records) from the IDs; the
  // last CTA also writes the routing arrays (the combine reads the inverse
  // permutation and scores from them, once every W2 tile is done)
  local_blocks(fa, reinterpret_cast<int*>(smem), reinterpret_cast<int4*>(cache), s_nblk);
  if (blockIdx.x == gridDim.x - 1) {
    fused_route(fa, reinterpret_cast<int*>(smem));   // the stage buffers are idle until the routing is out
    __syncthreads();
    if (threadIdx.x == 0) st_release_gpu(&sync[0], 1);   // cumulative over the CTA's stores (barrier above)
  }
  const int nblk = *s_nblk;
  const int n13 = fa.g13.n_tiles, n2 = fa.g2.n_tiles;
  const int gp = gather_parts(fa.D);
  const int U = nblk * (gp + n13 + n2) + fa.T * kCombineParts;
  MetaCache mc;
  mc.blocks = reinterpret_cast<const int4*>(cache);
  mc.poff = nullptr;
  mc.bstart = nullptr;
  int* s_route = reinterpret_cast<int*>(cache + kCacheBytes);   // [kBlockRows]: a gather record's routes

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < U; u += gridDim.x) {
      const Rec r = record(u, nblk, gp, n13, n2);
      if (r.kind != 1 && r.kind != 2) continue;
      const bool is13 = r.kind == 1;
      const Tile t = tile_of(fa, r, mc);
      const GemmParams& p = is13 ? fa.g13 : fa.g2;
      // the record's inputs: its block's gathered rows (W13) or its block's
      // h2 rows from all n13 W13 tiles (W2)
      int ready = 1;
      if (lane == 0) {
        // the block's gather first (a W13 tile's input; a W2 tile asks for
        // its weights no earlier, so the gathers' loads do not queue behind
        // weight traffic); a W2 tile whose W13 tiles are still running asks
        // L2 for its first kPrefetch weight stages and waits for them
        bool got = wait_counter(gather_done + r.b, gp, fa.wait_cycles, abort_flag, err);
        if (got && !is13 && ld_acquire_gpu(w13_done + r.b) < n13 + fa.stall) {
          for (int ks = 0; ks < min(kPrefetch, t.kstages); ++ks) tma_prefetch_l2_2d(&a2, ks * CF::BK, t.a_row[0]);
          got = wait_counter(w13_done + r.b, n13 + fa.stall, fa.wait_cycles, abort_flag, err);
        }
        // the acquires before this thread's tensor loads of what they guard
        fence_proxy_async_global();
        ready = got ? 1 : 0;
      }
      if (!__shfl_sync(0xFFFFFFFFu, ready, 0)) {
        ok = false;
        break;
      }
      for (int ks = 0; ks < t.kstages; ++ks, ++it) {
        const uint32_t slot = it % S, ph = (it / S) & 1;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&empty[slot], ph ^ 1, abort_flag, err))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* sa = smem + slot * CF::STAGE;
          uint8_t* sb = sa + 2 * kABytes;
          uint8_t* ssf = sb + kBBytes;
          mbar_arrive_expect_tx(&full[slot], (2 * 128 + t.b_rows) * 128 + CF::SF_BYTES);
          const int kx = ks * CF::BK;
          // the weight boxes kPrefetch stages ahead go to L2 now, so the
          // loads that will fetch them wait for L2, not HBM: one SM's loads
          // in flight bound its weight stream when few tiles share the GPU
          if (ks + kPrefetch < t.kstages) {
            const int px = kx + kPrefetch * CF::BK;
            if (is13) tma_prefetch_l2_3d(&a13, px, t.out_col0, 2 * t.e);
            else tma_prefetch_l2_2d(&a2, px, t.a_row[0]);
          }
          if (is13) {
            tma_load_3d(sa, &a13, &full[slot], kx, t.out_col0, 2 * t.e);   // gate, then up
            tma_load_4d(ssf, &sf13, &full[slot], 0, ks, t.out_col0 >> 7, 2 * t.e);
          } else {
            tma_load_2d(sa, &a2, &full[slot], kx, t.a_row[0]);            // two adjacent 128-row tiles
            tma_load_3d(ssf, &sf2, &full[slot], 0, ks, t.a_row[0] >> 7);
          }
          const CUtensorMap* b32 = is13 ? &bx32 : &bh32;
          if (t.b_rows == 128) {
            tma_load_2d(sb, is13 ? &bx128 : &bh128, &full[slot], kx, t.b_row0);
          } else {
            for (int c = 0; c < t.b_rows / 32; ++c) tma_load_2d(sb + c * 32 * 128, b32, &full[slot], kx, t.b_row0 + 32 * c);
          }
          bulk_load(ssf + 2 * kAtom, p.sfb + (t.sfb_atom + ks) * kAtom, kAtom, &full[slot]);
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      const uint32_t pend = it < static_cast<uint32_t>(S) ? it : static_cast<uint32_t>(S);
      for (uint32_t j = 0; j < pend; ++j) {
        const uint32_t i2 = it - 1 - j;
        drain_wait(&full[i2 % S], (i2 / S) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    uint32_t it = 0, tc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < U; u += gridDim.x) {
      const Rec r = record(u, nblk, gp, n13, n2);
      if (r.kind != 1 && r.kind != 2) continue;
      const Tile t = tile_of(fa, r, mc);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(tempty, (tc & 1) ^ 1, abort_flag, err))) break;
      tc_fence_after();
      const uint32_t idesc = idesc_mxf8(t.b_rows, 0, 0);
      for (int ks = 0; ks < t.kstages; ++ks, ++it) {
        const uint32_t slot = it % S, ph = (it / S) & 1;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[slot], ph, abort_flag, err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + slot * CF::STAGE);
        const uint32_t sb = sa + 2 * kABytes;
        const uint32_t sfcol = tmem + CF::SF_COL0 + slot * CF::SF_COLS;
        const uint64_t bdesc0 = sdesc_k_sw128(sb);
        const uint64_t adesc0[2] = {sdesc_k_sw128(sa), sdesc_k_sw128(sa + kABytes)};
        if (lane == 0) {
          // the stage's scale atoms go to its TMEM columns first (this
          // thread's tcgen05 operations run in order); the decode-sized
          // tiles this kernel serves are bound by how fast a stage cycles,
          // not by MMA issue
          const uint32_t ssf = sb + kBBytes;
#pragma unroll
          for (int j = 0; j <= 2; ++j) tc_cp_sf(sfcol + j * 4, sdesc_sf_atom(ssf + j * kAtom));
#pragma unroll
          for (int k = 0; k < CF::MMAS; ++k) {
            const uint64_t koff = static_cast<uint64_t>(2 * k);
            const uint32_t accum = (ks | k) ? 1u : 0u;
#pragma unroll
            for (int j = 0; j < 2; ++j)
              mma_mxf8(tmem + j * 128, adesc0[j] + koff, bdesc0 + koff,
                       idesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29), sfcol + j * 4,
                       sfcol + 8, accum);
          }
          tc_commit(&empty[slot]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc_commit(tfull);
      __syncwarp();
      ++tc;
    }
    if (lane == 0) {
      tc_commit(drain);
      drain_wait(drain, 0);
    }
    __syncwarp();
  } else if (warp == 2 + CF::EPI_WARPS) {
    // (the MMA thread copies the scale atoms itself here: this warp idles)
  } else {
    // -------------------------------------------- epilogue warps (8)
    // Every epilogue warp walks every record and reaches the end-of-record
    // barrier once per record, whether its own waits succeeded or not, so
    // a warp that gives up cannot leave the others blocked: they all see
    // the flag and leave together.
    const int ew = warp - 2;
    const int q = warp & 3;
    const int h = ew >> 2;
    const int lrow = q * 32 + lane;
    const int gtid = threadIdx.x - 64;
    uint32_t tc = 0;
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
      const Rec r = record(u, nblk, gp, n13, n2);
      bool ok = true;
      if (r.kind == 1 || r.kind == 2) {
        const Tile t = tile_of(fa, r, mc);
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(tfull, tc & 1, abort_flag, err));
        if (ok) {
          tc_fence_after();
          const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16);
          if (r.kind == 1) epi_swiglu_fwd<true>(fa.g13, t, tbase, lrow, lane, h, tempty);
          else epi_store<2>(fa.g2, t, tbase, lrow, lane, h, tempty);
        }
        ++tc;
      } else if (r.kind == 0) {
        const int4 blk = mc.blocks[r.b];   // nblk < kCacheBlocks (checked on the host)
        fused_gather(fa, r.b, r.n, gp, blk, gtid, s_route);
      } else {
        if (gtid == 0 && (!wait_counter(&sync[2], nblk * n2, fa.wait_cycles, abort_flag, err) ||
                          !wait_counter(&sync[0], 1, fa.wait_cycles, abort_flag, err)))
          *epi_abort = 1;
        named_bar_sync(kEpiBarrier, kEpiThreads);
        if (*epi_abort) break;
        fused_combine(fa, r.b, gtid);
      }
      if (!ok && lane == 0) *epi_abort = 1;
      fence_proxy_async_global();   // this record's stores, before their release below
      named_bar_sync(kEpiBarrier, kEpiThreads);
      if (*epi_abort) break;
      // the release is cumulative: it covers every epilogue thread's stores,
      // ordered before it by the barrier above
      if (gtid == 0 && r.kind != 3) {
        red_add_release_gpu(r.kind == 0 ? gather_done + r.b : (r.kind == 1 ? w13_done + r.b : &sync[2]), 1);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // the last CTA to finish returns every counter of this launch to zero for
  // the next one (every other CTA is past its last use of them)
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&sync[1], 1) == static_cast<int>(gridDim.x) - 1) {
      for (int b = 0; b < nblk; ++b) {
        gather_done[b] = 0;
        w13_done[b] = 0;
      }
      sync[0] = 0;
      sync[2] = 0;
      sync[1] = 0;
      __threadfence();
    }
  }
}

}  // namespace

cudaError_t launch_fused_forward(const FusedLaunch& L, int num_sms, cudaStream_t stream) {
  static PerDeviceOnce setup;
  const cudaError_t se = setup.once(
      [] { return cudaFuncSetAttribute(fused_forward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmem); });
  if (se != cudaSuccess) return se;
  const FusedArgs& fa = L.args;
  const long long recs =
      static_cast<long long>(L.max_blocks) * (gather_parts(fa.D) + fa.g13.n_tiles + fa.g2.n_tiles) +
      static_cast<long long>(fa.T) * kCombineParts;
  const int grid = static_cast<int>(std::max(1LL, std::min<long long>(num_sms, recs)));
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = kFusedSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident at once (the records wait on one another)
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_forward_kernel, L.a13, L.sf13, L.bx32, L.bx128, L.a2, L.sf2, L.bh32, L.bh128,
                            fa);
}

}  // namespace moe
