// Single-launch inference forward (MXFP8): routing, gather, W13 + SwiGLU,
// W2 and combine in one persistent grid.
//
// "Dist-MoE: Speed-of-light distributed Mixture-of-Experts kernels", section
// 05, "Kernel Pipelines: Staged and Mega": the staged forward runs ordered
// launches; the Mega forward joins W13 and W2 in one grid whose resident
// CTAs repeat work records on fixed warp roles (the same TMA, MMA and
// epilogue roles serve W13 and W2) and coordinate through readiness
// counters in global memory.  Here the grid also takes the routing (first,
// on CTA 0), the gather and the combine, so a decode-sized step is one
// launch.  "Mixture of Experts: How Routing Becomes GPU Computation",
// section 6: with few tokens, W13 has too few output tiles to fill the GPU;
// the CTAs that hold W2 tiles ask L2 for their weight slabs while the W13
// tiles they depend on are still running, so the W2 weights stream beside
// W13's instead of after them.
//
// Work records, numbered once the routing is known (nblk row blocks):
//   [0, nblk)                      gather block b (x rows -> MXFP8 row bundle)
//   [nblk, nblk (1 + n13))         W13 + SwiGLU tile (b, n), block-major
//   [.., + nblk n2)                W2 tile (b, n), block-major
//   [.., + T)                      combine token t
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
// Counters (ints in the context's scratch, zero between launches):
//   [0] routing published   [1] CTAs finished   [2] W2 tiles finished
//   [3 + b]                 gather of block b finished
//   [3 + b_cap + b]         W13 tiles of block b finished
// CTA 0 zeroes the per-block words and [2] before it publishes the routing;
// the last CTA to finish returns [0] and [1] to zero for the next launch.
#include <algorithm>

#include "gemm_core.cuh"

namespace moe {

namespace {

using CF = Cfg<true, 2, kGroupedM>;
constexpr int kFusedThreads = CF::THREADS;     // producer, MMA, 8 epilogue warps, scale copier
constexpr int kEpiThreads = CF::EPI_THREADS;

struct Rec {
  int kind;   // 0 gather, 1 W13 tile, 2 W2 tile, 3 combine
  int b, n;   // block and slice (tiles), block (gather), token (combine: b)
};

__device__ __forceinline__ Rec record(int u, int nblk, int n13, int n2) {
  Rec r{};
  if (u < nblk) {
    r.kind = 0;
    r.b = u;
    return r;
  }
  u -= nblk;
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

// ------------------------------------------------------------------ routing
// CTA 0, all threads: the same arrays as the routing kernel (counts,
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
// The 8 epilogue warps, one row at a time each: the row bundle of the
// block's rows exactly as the inference gather writes it (4 lanes per
// 32-value block, E8M0 scale into the block's atoms, pad rows zero).
__device__ void fused_gather(const FusedArgs& fa, int b, const int4 blk, int ew, int lane) {
  const int D = fa.D, K = fa.K;
  const long long atom_row = static_cast<long long>(b) * (D / 128);
  for (int r = blk.y + ew; r < blk.y + blk.z; r += CF::EPI_WARPS) {
    const int route = __ldcg(fa.rp.perm + r);
    const __nv_bfloat16* srow = route >= 0 ? fa.x + static_cast<long long>(route / K) * D : nullptr;
    const int p = r - blk.y;
    for (int base = 0; base < D; base += 1024) {
      uint4 ub[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int cq = base + q * 256 + lane * 8;
        ub[q] = make_uint4(0, 0, 0, 0);
        if (cq < D && srow) ub[q] = __ldg(reinterpret_cast<const uint4*>(srow + cq));
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = base + q * 256 + lane * 8;
        const uint4 u = ub[q];
        float v[8] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y),
                      bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w)};
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        const int e = mx_shared_exp(amax);
        const float inv = exp2_int(-e);
        uint2 qv;
        qv.x = cvt_e4m3x2(v[0] * inv, v[1] * inv) | (cvt_e4m3x2(v[2] * inv, v[3] * inv) << 16);
        qv.y = cvt_e4m3x2(v[4] * inv, v[5] * inv) | (cvt_e4m3x2(v[6] * inv, v[7] * inv) << 16);
        if (c < D) {
          *reinterpret_cast<uint2*>(fa.xrow + static_cast<long long>(r) * D + c) = qv;
          if ((lane & 3) == 0) {
            const int kb = c >> 5;
            fa.xsf[(atom_row + (kb >> 2)) * 512 + sf_atom_byte(p, kb & 3)] = static_cast<uint8_t>(e + 127);
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------ combine token
// out[t] = bf16((accumulate ? out[t] : 0) + sum_k s h3[inv]) in FP32, k in
// order: the combine kernel's arithmetic, with h3 read through L2 (other
// CTAs wrote it in this launch).
__device__ void fused_combine(const FusedArgs& fa, int t, int gtid) {
  const int D = fa.D, K = fa.K;
  __nv_bfloat16* orow = fa.out + static_cast<long long>(t) * D;
  const __nv_bfloat16* h3 = static_cast<const __nv_bfloat16*>(fa.g2.out0);
  for (int c = gtid * 8; c < D; c += kEpiThreads * 8) {
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
    for (int k = 0; k < K; ++k) {
      const int r = __ldcg(fa.rp.inv + t * K + k);
      if (r < 0) continue;
      const float s = __ldcg(fa.rp.scores + t * K + k);
      const uint4 u = __ldcg(reinterpret_cast<const uint4*>(h3 + static_cast<long long>(r) * D + c));
      acc[0] = fmaf(s, bf16_lo(u.x), acc[0]);
      acc[1] = fmaf(s, bf16_hi(u.x), acc[1]);
      acc[2] = fmaf(s, bf16_lo(u.y), acc[2]);
      acc[3] = fmaf(s, bf16_hi(u.y), acc[3]);
      acc[4] = fmaf(s, bf16_lo(u.z), acc[4]);
      acc[5] = fmaf(s, bf16_hi(u.z), acc[5]);
      acc[6] = fmaf(s, bf16_lo(u.w), acc[6]);
      acc[7] = fmaf(s, bf16_hi(u.w), acc[7]);
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
  uint64_t* sf_full = drain + 1;   // [S]
  uint64_t* sf_drain = sf_full + S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_drain + 1);
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
      mbar_init(&sf_full[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, CF::EPI_WARPS);
    mbar_init(drain, 1);
    mbar_init(sf_drain, 1);
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

  // ---- routing (CTA 0), then every CTA waits for it to be published
  if (blockIdx.x == 0) {
    fused_route(fa, reinterpret_cast<int*>(smem));   // the stage buffers are idle until the routing is out
    __syncthreads();
    if (threadIdx.x == 0) {
      const int nb = fa.rp.hdr[1];
      for (int b = 0; b < nb; ++b) {
        gather_done[b] = 0;
        w13_done[b] = 0;
      }
      sync[2] = 0;
      __threadfence();
      st_release_gpu(&sync[0], 1);
    }
  }
  if (threadIdx.x == 0) {
    if (wait_counter(&sync[0], 1, fa.wait_cycles, abort_flag, err)) *s_nblk = __ldcg(fa.rp.hdr + 1);
  }
  __syncthreads();
  const int nblk = *s_nblk;
  const int n13 = fa.g13.n_tiles, n2 = fa.g2.n_tiles;
  const int U = *abort_flag ? 0 : nblk * (1 + n13 + n2) + fa.T;
  MetaCache mc;
  mc.blocks = reinterpret_cast<const int4*>(cache);
  mc.poff = nullptr;
  mc.bstart = nullptr;
  {
    int4* sb = reinterpret_cast<int4*>(cache);
    for (int i = threadIdx.x; i < min(nblk, kCacheBlocks); i += blockDim.x) sb[i] = __ldcg(fa.rp.blocks + i);
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < U; u += gridDim.x) {
      const Rec r = record(u, nblk, n13, n2);
      if (r.kind != 1 && r.kind != 2) continue;
      const bool is13 = r.kind == 1;
      const Tile t = tile_of(fa, r, mc);
      const GemmParams& p = is13 ? fa.g13 : fa.g2;
      // the record's inputs: its block's gathered rows (W13) or its block's
      // h2 rows from all n13 W13 tiles (W2)
      int ready = 1;
      if (lane == 0) {
        const int* dep = is13 ? gather_done + r.b : w13_done + r.b;
        const int need = is13 ? 1 : n13 + fa.stall;
        if (!is13 && ld_acquire_gpu(dep) < need) {
          // while waiting, have L2 fetch this tile's two weight slabs (256
          // adjacent rows of F bytes) and their scale atoms
          const uint8_t* slab = fa.w2 + static_cast<long long>(t.a_row[0]) * p.K;
          const uint32_t bytes = 256u * static_cast<uint32_t>(p.K);
          for (uint32_t o = 0; o < bytes; o += 32768u) prefetch_l2(slab + o, min(32768u, bytes - o));
          prefetch_l2(p.sfa + t.sfa_atom[0] * kAtom, static_cast<uint32_t>(2 * p.sfa_ts * kAtom));
        }
        ready = wait_counter(dep, need, fa.wait_cycles, abort_flag, err) ? 1 : 0;
        fence_proxy_async_global();
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
      const Rec r = record(u, nblk, n13, n2);
      if (r.kind != 1 && r.kind != 2) continue;
      const Tile t = tile_of(fa, r, mc);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(tempty, (tc & 1) ^ 1, abort_flag, err))) break;
      tc_fence_after();
      const uint32_t idesc = idesc_mxf8(t.b_rows, 0, 0);
      for (int ks = 0; ks < t.kstages; ++ks, ++it) {
        const uint32_t slot = it % S, ph = (it / S) & 1;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sf_full[slot], ph, abort_flag, err))) {
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
    // ------------------------------------------------- scale-atom copier
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < U; u += gridDim.x) {
      const Rec r = record(u, nblk, n13, n2);
      if (r.kind != 1 && r.kind != 2) continue;
      const Tile t = tile_of(fa, r, mc);
      for (int ks = 0; ks < t.kstages; ++ks, ++it) {
        const uint32_t slot = it % S, ph = (it / S) & 1;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[slot], ph, abort_flag, err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sfcol = tmem + CF::SF_COL0 + slot * CF::SF_COLS;
          const uint32_t ssf = smem_u32(smem + slot * CF::STAGE) + 2 * kABytes + kBBytes;
#pragma unroll
          for (int j = 0; j <= 2; ++j) tc_cp_sf(sfcol + j * 4, sdesc_sf_atom(ssf + j * kAtom));
          tc_commit(&sf_full[slot]);
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      tc_commit(sf_drain);
      drain_wait(sf_drain, 0);
    }
    __syncwarp();
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
      const Rec r = record(u, nblk, n13, n2);
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
        const int4 blk = r.b < kCacheBlocks ? mc.blocks[r.b] : __ldcg(fa.rp.blocks + r.b);
        fused_gather(fa, r.b, blk, ew, lane);
      } else {
        if (gtid == 0 && !wait_counter(&sync[2], nblk * n2, fa.wait_cycles, abort_flag, err)) *epi_abort = 1;
        named_bar_sync(kEpiBarrier, kEpiThreads);
        if (*epi_abort) break;
        fused_combine(fa, r.b, gtid);
      }
      if (!ok && lane == 0) *epi_abort = 1;
      fence_proxy_async_global();   // this record's stores, before their release below
      named_bar_sync(kEpiBarrier, kEpiThreads);
      if (*epi_abort) break;
      if (gtid == 0 && r.kind != 3) {
        __threadfence();
        if (r.kind == 0) st_release_gpu(gather_done + r.b, 1);
        else red_add_release_gpu(r.kind == 1 ? w13_done + r.b : &sync[2], 1);
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
  // the last CTA to finish returns the routing flag to zero for the next
  // launch (every CTA read it, once, at its start)
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&sync[1], 1) == static_cast<int>(gridDim.x) - 1) {
      sync[0] = 0;
      sync[1] = 0;
      __threadfence();
    }
  }
}

}  // namespace

cudaError_t launch_fused_forward(const FusedLaunch& L, int num_sms, cudaStream_t stream) {
  static PerDeviceOnce setup;
  const cudaError_t se = setup.once(
      [] { return cudaFuncSetAttribute(fused_forward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM); });
  if (se != cudaSuccess) return se;
  const FusedArgs& fa = L.args;
  const long long recs = static_cast<long long>(L.max_blocks) * (1 + fa.g13.n_tiles + fa.g2.n_tiles) + fa.T;
  const int grid = static_cast<int>(std::max(1LL, std::min<long long>(num_sms, recs)));
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = CF::SMEM;
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
