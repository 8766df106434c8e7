// Grouped GEMMs of the MoE layer on the 5th-generation tensor cores
// (tcgen05.mma, FP32 accumulators in tensor memory, operands staged by TMA).
//
// "Mixture of Experts: How Routing Becomes GPU Computation", section 2,
// "Grouped GEMM": each expert e computes C_e = A_e B_e^T over its own ragged
// row range, with weights stacked [E, N, K]; "Grouped GEMM backward":
// dA_e = dC_e B_e and dB_e = dC_e^T A_e.  Dist-MoE explainer section 05,
// "GPU Kernels: Tiles and Warp Roles": a persistent scheduler hands each CTA
// an expert's row/output tile, TMA stages operand tiles into shared memory,
// MMA accumulates in FP32 tensor memory, and an epilogue drains it; tails are
// masked.
//
// Two ways of walking the experts:
//  * grouped-M (forward W13 and W2, input-gradient DGRAD): the weight is the
//    A operand (128 output features per tile, M = 128) and one routing row
//    block of the expert (32..128 rows) is the B operand (N = its rows).
//    Experts get only ~32 rows at the 384-expert shape, so putting weights
//    on the 128-wide M side keeps the MMA from computing padding and reads
//    each weight tile once per row block.
//  * grouped-M over row-block pairs (kGroupedMP), for routings dense enough
//    that experts have two or more blocks: B is two consecutive blocks of
//    one expert (N up to 256).  A tensor-core instruction of N = 128 takes
//    about as long as one of N = 256 on this part, so at the compute-bound
//    shapes 256-wide instructions double the rate.  One A tile of 128 rows
//    per stage (a 256-column accumulator: single-buffered in MXFP8, whose
//    scale columns need the rest of TMEM); the SwiGLU forward's A tile is 64
//    gate rows followed by the 64 up rows of the same features, and its
//    epilogue pairs them up through shared memory.
//  * the same pair tiles on CTA pairs (kGroupedMC): a cluster of two
//    CTAs on two SMs takes two adjacent A tiles (SwiGLU: features f..f+63
//    and f+64..f+127) against one row-block pair, each CTA loading its own
//    A tile and one block of the pair.  The lower-ranked CTA issues one
//    tcgen05.mma.cta_group::2 of M = 256, N = 256 per K step over both; each
//    CTA's 128 accumulator lanes hold its A tile's rows against all 256
//    columns, and each CTA drains its own.  Per SM a stage then carries 32 KB
//    of operands instead of 48 for the same tensor-core work (stages hold two
//    K-chunks: 64 KB per SM; BF16 double-buffers the accumulator, having no
//    scale columns in TMEM).  Rank 1 reports
//    each stage's operands in place (and each accumulator drained) to rank 0
//    through mbarriers in rank 0's shared memory; rank 0's commits release
//    the stages and hand over the accumulators in both CTAs (multicast).
//  * grouped-K (WGRAD): dW_e[m, n] = sum over the expert's rows of
//    colA[m, r] colB[n, r]; both operands are column bundles stored
//    [features, rows], so the contraction runs over the expert's row range.
//
// MXFP8 scales travel with the operand tiles: the TMA producer copies one
// 512-byte scale atom per operand per stage into the stage's shared memory
// (the one-A-tile grouped-M GEMMs: four stages' atoms per copy, into a ring
// of their own), a scale warp moves them to tensor memory with tcgen05.cp
// and commits them to the stage's sf_full barrier, and the MMA thread,
// which waits on that barrier, issues the block-scaled MMAs.  On CTA pairs
// the MMA thread issues the copies itself, just before the stage's MMAs (a
// copy and the MMAs after it from one thread run in issue order with no
// wait between them, and next to 256-wide MMAs the copies cost no tensor
// time), so the stage's chain has one hop less.
//
// Epilogues: fused SwiGLU forward (h1 -> h2 row/column bundles), plain BF16
// store (h3, input-gradient rows), fused SwiGLU backward (dh2 -> dh1 row and
// column bundles) and weight-gradient store (BF16 through shared memory and
// TMA; FP32 or accumulate with plain stores).
//
// Warp roles (one CTA per SM, persistent over tiles; warps 0, 1 and the
// scale warp run their loops converged and lane 0 issues):
//   warp 0      TMA producer
//   warp 1      TMEM allocator and MMA issuer (CTA pairs, rank 1: tells
//               rank 0 when its epilogue has drained the accumulator)
//   warps 2..9  epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 and the
//               32-column chunks 32h and 32h + 64 (h = (w-2)/4) of the
//               accumulator
//   warps 10..17  weight gradient only: a second epilogue group of 8 warps;
//               the two groups take alternate tiles
//   last warp   MXFP8 (and BF16 on CTA pairs): copies the scale atoms, or
//               over row-block pairs builds the SwiGLU forward's weight atom
//               of each stage; CTA pairs: tells rank 0's MMA thread when a
//               stage's operands are in place
#include "gemm_core.cuh"

namespace moe {

namespace {

// DWF (weight gradient only): the FP32 staged modes (TMA store or TMA
// reduce-add) are compiled into this instance; the other instance holds the
// BF16 staged store and the plain-store epilogue, so neither carries the
// other's registers.
template <bool MX, int NA, int EPI, int MODE, bool DWF = false>
__global__ void __launch_bounds__(Cfg<MX, NA, MODE>::THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap aux0,
                const __grid_constant__ CUtensorMap aux1, const __grid_constant__ CUtensorMap aux2,
                const __grid_constant__ CUtensorMap aux3, const GemmParams p) {
  using C = Cfg<MX, NA, MODE>;
  constexpr int S = C::S;
  constexpr bool PAIR = C::PAIR;
  constexpr bool CG2 = C::CG2;
  constexpr int CG = CG2 ? 2 : 1;
  constexpr int kStep = PAIR ? (EPI == kEpiSwigluFwd ? 64 : 128) : ((NA == 2 && EPI != kEpiSwigluFwd) ? 256 : 128);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + S * C::STAGE;
  uint8_t* sfg = staging + C::STAGING;     // [SFR][GROUP_BYTES]: scale-atom groups (SFG)
  uint8_t* xbuf = sfg + C::SFG_BYTES;      // [EXCH]: the pair SwiGLU epilogue's exchange
  uint64_t* full = reinterpret_cast<uint64_t*>(xbuf + C::EXCH);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + C::ACC_BUFS;
  uint64_t* drain = tempty + C::ACC_BUFS;
  uint64_t* sf_full = drain + 1;            // [S]: a stage's scale atoms are in TMEM (MXFP8)
  uint64_t* sf_drain = sf_full + S;
  uint64_t* sfg_full = sf_drain + 1;        // [SFR]: a scale-atom group has landed
  uint64_t* sfg_empty = sfg_full + C::SFR;  // [SFR]: its atoms are in TMEM
  uint64_t* ready = sfg_empty + C::SFR;     // CTA pairs [S]: both CTAs' operands of a stage are in place
  uint64_t* ptempty = ready + (CG2 ? S : 0);   // CTA pairs [ACC_BUFS]: the other CTA drained its accumulator
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ptempty + (CG2 ? C::ACC_BUFS : 0));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_abort = abort_flag + 1;  // [EPI_GROUPS]: a group's warps leave together
  uint8_t* cache = xbuf + C::EXCH + C::BARS;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA pairs: both CTAs of a cluster walk the same tiles (cluster index cid
  // of ncl), rank 0 issuing the MMAs for both
  const uint32_t rank = CG2 ? cluster_ctarank() : 0u;
  const int cid = CG2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int ncl = CG2 ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < C::ACC_BUFS; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], C::EPI_WARPS / C::EPI_GROUPS);
    }
    mbar_init(drain, 1);
    for (int s2 = 0; s2 < S; ++s2) mbar_init(&sf_full[s2], 1);
    mbar_init(sf_drain, 1);
    for (int g = 0; g < C::SFR; ++g) {
      mbar_init(&sfg_full[g], 1);
      mbar_init(&sfg_empty[g], 1);
    }
    if (CG2) {
      for (int s = 0; s < S; ++s) mbar_init(&ready[s], 2);
      for (int a = 0; a < C::ACC_BUFS; ++a) mbar_init(&ptempty[a], 1);
    }
    *abort_flag = 0;
    for (int g = 0; g < C::EPI_GROUPS; ++g) epi_abort[g] = 0;
    mbar_fence_init();
    tma_prefetch(&tmA);
    tma_prefetch(&tmB);
    if (C::WGRAD && p.tma_store) tma_prefetch(&tmC);
    if (C::WGRAD) {
      tma_prefetch(&aux0);
      tma_prefetch(&aux1);
      tma_prefetch(&aux2);
      tma_prefetch(&aux3);
    } else {
      if (p.a_pair_box) {
        tma_prefetch(&aux0);
        if (MX) tma_prefetch(&aux2);
      }
      if (p.b_full_box) tma_prefetch(&aux1);
    }
  }
  if (warp == 1) {
    // CTA pairs: one warp of each CTA together, the same columns in both
    tmem_alloc_cg<CG>(tmem_slot, 512);
    tmem_relinquish_cg<CG>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the other CTA's barriers are initialised before anything arrives on them
  if (CG2) cluster_sync();

  const int nblk = (MODE != kGroupedK) ? p.hdr[1] : 0;
  const int num_tiles = (MODE == kGroupedM)    ? nblk * p.n_tiles
                        : (MODE == kGroupedMP || MODE == kGroupedMC) ? p.hdr[4] * p.n_tiles
                                               : p.E * p.m_tiles * p.n_tiles;
  MetaCache mc;
  mc.blocks = reinterpret_cast<const int4*>(cache);
  mc.ncache = C::CACHE / 16;
  mc.poff = reinterpret_cast<const int*>(cache);
  mc.bstart = reinterpret_cast<const int*>(cache) + 1028;
  if (MODE != kGroupedK) {
    int4* sb = reinterpret_cast<int4*>(cache);
    for (int i = threadIdx.x; i < min(nblk, mc.ncache); i += blockDim.x) sb[i] = p.blocks[i];
  } else {
    int* sp = reinterpret_cast<int*>(cache);
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
      sp[i] = p.poffsets[i];
      sp[1028 + i] = (p.bstart != nullptr) ? p.bstart[i] : 0;
    }
  }
  __syncthreads();
  // A tile of the walk; CTA pairs: this CTA's half (A tile 2n + rank)
  auto tile_at = [&](TileWalk<MODE> w) {
    if (CG2) w.n = 2 * w.n + static_cast<int>(rank);
    return decode_tile<MODE, C::BK, kStep>(p, w, mc);
  };

  // The producer and MMA warps walk their loops with all 32 lanes, so the
  // loop state and the descriptors stay warp-uniform; lane 0 alone issues
  // the copies and the tensor-core instructions (and the commits, which
  // track the issuing thread's operations).
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    uint32_t it = 0, gc = 0;   // gc: scale-atom groups issued (SFG)
    bool ok = true;
    TileWalk<MODE> w;
    w.start(p, cid);
    for (; ok && w.tile < num_tiles; w.advance(p)) {
      const Tile t = tile_at(w);
      for (int ks = 0; ks < t.kstages; ++ks, ++it) {
        const uint32_t slot = it % S, ph = (it / S) & 1;
        if (C::SFG && ks % C::GS == 0) {
          // the group's atoms (weight, then row block), once the scale warp
          // has moved the group that last used the buffer into TMEM
          const uint32_t g = gc % C::SFR, gph = (gc / C::SFR) & 1;
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sfg_empty[g], gph ^ 1, abort_flag, p.err))) {
            ok = false;
            break;
          }
          if (lane == 0) {
            const int n = min(C::GS, t.kstages - ks);
            uint8_t* dst = sfg + g * C::GROUP_BYTES;
            mbar_arrive_expect_tx(&sfg_full[g], 2 * n * kAtom);
            bulk_load(dst, p.sfa + (t.sfa_atom[0] + ks) * kAtom, n * kAtom, &sfg_full[g]);
            bulk_load(dst + C::GS * kAtom, p.sfb + (t.sfb_atom + ks) * kAtom, n * kAtom, &sfg_full[g]);
          }
          ++gc;
        }
        if (!__all_sync(0xFFFFFFFFu, mbar_wait<CG2>(&empty[slot], ph ^ 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* sa = smem + slot * C::STAGE;
          uint8_t* sb = sa + C::A_BYTES;
          uint8_t* ssf = sa + C::SF_OFF;
          const int rb = stage_row_bytes<MODE, C::BK, MX ? 1 : 2>(t, ks);
          const int kx = t.k0 + ks * C::BK;
          if (CG2) {
            // two K-chunks (kc, kc + 1): the A tile (SwiGLU: gate and up
            // halves) and this CTA's block of the pair in one box each (none
            // for rank 1 of a lone block), the weight's atoms of both chunks
            // (SwiGLU: of both halves) at ssf, then each block's two atoms
            const bool two = t.b_rows > 128;
            const bool mine = rank == 0 || two;
            const int kc = kx / (MX ? 128 : 64);   // 128-byte chunks
            mbar_arrive_expect_tx(&full[slot], C::A_BYTES + (mine ? C::B_BYTES : 0) +
                                                   (MX ? ((EPI == kEpiSwigluFwd ? 4 : 2) + (two ? 4 : 2)) * kAtom : 0));
            if (EPI == kEpiSwigluFwd) tma_load_4d(sa, &aux0, &full[slot], 0, t.out_col0, 2 * t.e, kc);
            else tma_load_3d(sa, &aux0, &full[slot], 0, t.a_row[0], kc);
            if (mine) tma_load_3d(sb, &aux1, &full[slot], 0, t.b_row0 + 128 * static_cast<int>(rank), kc);
            if (MX) {
              if (EPI == kEpiSwigluFwd) tma_load_4d(ssf, &aux2, &full[slot], 0, kc, t.out_col0 >> 7, 2 * t.e);
              else bulk_load(ssf, p.sfa + (t.sfa_atom[0] + kc) * kAtom, 2 * kAtom, &full[slot]);
              bulk_load(ssf + 4 * kAtom, p.sfb + (t.sfb_atom + kc) * kAtom, 2 * kAtom, &full[slot]);
              if (two)
                bulk_load(ssf + 6 * kAtom, p.sfb + (t.sfb_atom + p.sfb_ts + kc) * kAtom, 2 * kAtom, &full[slot]);
            }
          } else if (PAIR) {
            // one A tile (SwiGLU: its gate and up halves in one 3D box), B as
            // full 128-row boxes then 32-row boxes; MXFP8: the weight's atom
            // (two for the halves) and one atom per routing block of the pair
            const bool two = t.b_rows > 128;
            mbar_arrive_expect_tx(&full[slot], (128 + t.b_rows) * rb +
                                                   (MX ? ((EPI == kEpiSwigluFwd ? 2 : 1) + (two ? 2 : 1)) * kAtom : 0));
            if (EPI == kEpiSwigluFwd) tma_load_3d(sa, &aux0, &full[slot], kx, t.out_col0, 2 * t.e);
            else if (MX && p.a_mn) tma_load_2d(sa, &tmA, &full[slot], t.a_row[0] - t.e * p.a_rows_per_expert, t.e * p.K + kx);
            else tma_load_2d(sa, &tmA, &full[slot], kx, t.a_row[0]);
            int r = 0;
            if (p.b_full_box)
              for (; r + 128 <= t.b_rows; r += 128) tma_load_2d(sb + r * 128, &aux1, &full[slot], kx, t.b_row0 + r);
            for (; r < t.b_rows; r += 32) tma_load_2d(sb + r * 128, &tmB, &full[slot], kx, t.b_row0 + r);
            if (MX) {
              if (EPI == kEpiSwigluFwd) tma_load_4d(ssf, &aux2, &full[slot], 0, ks, t.out_col0 >> 7, 2 * t.e);
              else bulk_load(ssf, p.sfa + (t.sfa_atom[0] + ks) * kAtom, kAtom, &full[slot]);
              bulk_load(ssf + 2 * kAtom, p.sfb + (t.sfb_atom + ks) * kAtom, kAtom, &full[slot]);
              if (two) bulk_load(ssf + 3 * kAtom, p.sfb + (t.sfb_atom + p.sfb_ts + ks) * kAtom, kAtom, &full[slot]);
            }
          } else {
          mbar_arrive_expect_tx(&full[slot], (NA * 128 + t.b_rows) * rb + (C::SFG ? 0 : C::SF_BYTES));
          if (MODE == kGroupedK) {
            const CUtensorMap* ta = rb == 128 ? &tmA : (rb == 64 ? &aux0 : &aux2);
            const CUtensorMap* tb = rb == 128 ? &tmB : (rb == 64 ? &aux1 : &aux3);
#pragma unroll
            for (int j = 0; j < NA; ++j) tma_load_2d(sa + j * kABytes, ta, &full[slot], kx, t.a_row[j]);
            for (int c = 0; c < t.b_rows / p.b_box_rows; ++c)
              tma_load_2d(sb + c * p.b_box_rows * rb, tb, &full[slot], kx, t.b_row0 + p.b_box_rows * c);
          } else {
            // fewer, larger copies: the issue rate of the producer thread
            // bounds compute-bound shapes
            if (MX && p.a_mn) {
              // MN-major A: box (M columns of this tile, K rows of this
              // stage) of the weight as prepared for the forward, [E * K, M]
#pragma unroll
              for (int j = 0; j < NA; ++j)
                tma_load_2d(sa + j * kABytes, &tmA, &full[slot], t.a_row[j] - t.e * p.a_rows_per_expert,
                            t.e * p.K + kx);
            } else if (NA == 2 && p.a_pair_box == 1) {
              tma_load_2d(sa, &aux0, &full[slot], kx, t.a_row[0]);   // rows a_row[0] .. +255
            } else if (NA == 2 && p.a_pair_box == 2) {
              tma_load_3d(sa, &aux0, &full[slot], kx, t.out_col0, 2 * t.e);   // gate, then up
            } else {
#pragma unroll
              for (int j = 0; j < NA; ++j) tma_load_2d(sa + j * kABytes, &tmA, &full[slot], kx, t.a_row[j]);
            }
            if (t.b_rows == 128 && p.b_full_box) {
              tma_load_2d(sb, &aux1, &full[slot], kx, t.b_row0);
            } else {
              for (int c = 0; c < t.b_rows / p.b_box_rows; ++c)
                tma_load_2d(sb + c * p.b_box_rows * 128, &tmB, &full[slot], kx, t.b_row0 + p.b_box_rows * c);
            }
          }
          if (MX && !C::SFG) {
            if (MODE == kGroupedM && NA == 2 && p.a_pair_box == 1) {
              tma_load_3d(ssf, &aux2, &full[slot], 0, ks, t.a_row[0] >> 7);
            } else if (MODE == kGroupedM && NA == 2 && p.a_pair_box == 2) {
              tma_load_4d(ssf, &aux2, &full[slot], 0, ks, t.out_col0 >> 7, 2 * t.e);
            } else {
#pragma unroll
              for (int j = 0; j < NA; ++j)
                bulk_load(ssf + j * kAtom, p.sfa + (t.sfa_atom[j] + ks) * kAtom, kAtom, &full[slot]);
            }
            bulk_load(ssf + NA * kAtom, p.sfb + (t.sfb_atom + ks) * kAtom, kAtom, &full[slot]);
          }
          }
        }
        __syncwarp();
      }
    }
    // no load may still be landing in shared memory when the CTA exits
    if (lane == 0) {
      const uint32_t pend = it < static_cast<uint32_t>(S) ? it : static_cast<uint32_t>(S);
      for (uint32_t j = 0; j < pend; ++j) {
        const uint32_t i2 = it - 1 - j;
        drain_wait(&full[i2 % S], (i2 / S) & 1);
      }
      const uint32_t gpend = gc < static_cast<uint32_t>(C::SFR) ? gc : static_cast<uint32_t>(C::SFR);
      for (uint32_t j = 0; j < gpend; ++j) {
        const uint32_t i2 = gc - 1 - j;
        drain_wait(&sfg_full[i2 % C::SFR], (i2 / C::SFR) & 1);
      }
    }
    __syncwarp();
  } else if (CG2 && warp == 1 && rank != 0) {
    // ------------------------------------ CTA pairs, rank 1: accumulator relay
    // Rank 0's MMA thread reuses the accumulator once this CTA's epilogue
    // has drained its lanes as well.
    const uint32_t peer_ptempty = cluster_addr(ptempty, 0);
    uint32_t tc = 0;
    TileWalk<MODE> w;
    w.start(p, cid);
    for (; w.tile < num_tiles; w.advance(p), ++tc) {
      const uint32_t acc = tc % C::ACC_BUFS, aph = (tc / C::ACC_BUFS) & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait<true>(&tempty[acc], aph, abort_flag, p.err))) break;
      if (lane == 0) mbar_arrive_cluster(peer_ptempty + 8 * acc);
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    uint32_t it = 0, tc = 0;
    bool ok = true;
    TileWalk<MODE> w;
    w.start(p, cid);
    for (; ok && w.tile < num_tiles; w.advance(p), ++tc) {
      const Tile t = tile_at(w);
      const uint32_t acc = tc % C::ACC_BUFS, aph = (tc / C::ACC_BUFS) & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tempty[acc], aph ^ 1, abort_flag, p.err))) break;
      if (CG2 && !__all_sync(0xFFFFFFFFu, mbar_wait<true>(&ptempty[acc], aph ^ 1, abort_flag, p.err))) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem + acc * C::ACC_COLS;
      // CTA pairs: M = 256 over both CTAs and N = 256 (a lone block's other
      // half is whatever the other CTA's stage holds; its columns are never read)
      const uint32_t idesc = MX ? (idesc_mxf8(CG2 ? 256 : t.b_rows, 0, 0, CG2 ? 256 : 128) |
                                   (MODE != kGroupedK && p.a_mn ? kIdescAMnMajor : 0u))
                                : idesc_bf16(CG2 ? 256 : t.b_rows, CG2 ? 256 : 128);
      for (int ks = 0; ks < t.kstages; ++ks, ++it) {
        const uint32_t slot = it % S, ph = (it / S) & 1;
        // MXFP8: the scale warp's commit for this stage follows its own wait
        // for the stage's data, so it covers both.  CTA pairs: both CTAs'
        // scale warps report the stage in place (weight atom built), and this
        // thread copies the atoms itself, just before the stage's MMAs.
        uint64_t* in_place = CG2 ? &ready[slot] : (MX ? &sf_full[slot] : &full[slot]);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait<CG2>(in_place, ph, abort_flag, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + slot * C::STAGE);
        const uint32_t sb = sa + C::A_BYTES;
        const uint32_t sfcol = tmem + C::SF_COL0 + slot * C::SF_COLS;
        const int rb = stage_row_bytes<MODE, C::BK, MX ? 1 : 2>(t, ks);
        const uint64_t bdesc0 = sdesc_k_sw(sb, rb);
        // MN-major A (grouped-M MXFP8 with p.a_mn): a K step of 32 rows is 4 KB on
        const bool amn = MX && MODE != kGroupedK && p.a_mn;
        uint64_t adesc0[NA];
#pragma unroll
        for (int j = 0; j < NA; ++j) adesc0[j] = amn ? sdesc_mn_sw128(sa + j * kABytes) : sdesc_k_sw(sa + j * kABytes, rb);
        const uint64_t astep = amn ? (4096 >> 4) : 2;
        const int nmma = (ks == t.kstages - 1) ? t.klast / C::KMMA : C::MMAS;
        if (lane == 0 && CG2) {
          // per K-chunk c: the weight's atom, then the pair's B atoms (every
          // SM's MMA reads the scales of all 256 columns) into columns
          // 12c .. 12c + 11 of the stage, then the chunk's four MMAs
          const uint32_t ssf = sa + C::SF_OFF;
          const bool two = t.b_rows > 128;
#pragma unroll
          for (int c = 0; c < C::KCH; ++c) {
            const uint32_t sfc = sfcol + 12 * c;
            if (MX) {
              tc_cp_sf_pair(sfc, sdesc_sf_atom(ssf + c * kAtom));
              tc_cp_sf_pair(sfc + 4, sdesc_sf_atom(ssf + (4 + c) * kAtom));
              if (two) tc_cp_sf_pair(sfc + 8, sdesc_sf_atom(ssf + (6 + c) * kAtom));
            }
            const uint64_t ad = sdesc_k_sw(sa + c * kABytes, 128), bd = sdesc_k_sw(sb + c * kBBytes, 128);
#pragma unroll
            for (int k = 0; k < 4; ++k) {   // 32 bytes of K each (32 E4M3 or 16 BF16 values)
              if (MX)
                mma_mxf8_pair(d_tmem, ad + 2 * k, bd + 2 * k,
                              idesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29), sfc,
                              sfc + 4, (ks | c | k) ? 1u : 0u);
              else
                mma_bf16_pair(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (ks | c | k) ? 1u : 0u);
            }
          }
          // the stage is free in both CTAs
          tc_commit_pair_mc(&empty[slot], 3);
        } else if (lane == 0) {
#pragma unroll
          for (int k = 0; k < C::MMAS; ++k) {
            if (k < nmma) {
              const uint64_t koff = static_cast<uint64_t>(2 * k);   // +32 bytes along K
              const uint32_t accum = (ks | k) ? 1u : 0u;
#pragma unroll
              for (int j = 0; j < NA; ++j) {
                if (MX) {
                  // scale byte k of the 4 per row (one per 32-element block)
                  mma_mxf8(d_tmem + j * 128, adesc0[j] + static_cast<uint64_t>(k) * astep, bdesc0 + koff,
                           idesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29), sfcol + j * 4,
                           sfcol + NA * 4, accum);
                } else {
                  mma_bf16(d_tmem + j * 128, adesc0[j] + koff, bdesc0 + koff, idesc, accum);
                }
              }
            }
          }
          tc_commit(&empty[slot]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) {
        if (CG2) tc_commit_pair_mc(&tfull[acc], 3);
        else tc_commit(&tfull[acc]);
      }
      __syncwarp();
    }
    // every MMA (and scale copy) issued here must be complete before TMEM is released
    if (lane == 0) {
      if (CG2) tc_commit_pair(drain);
      else tc_commit(drain);
      drain_wait(drain, 0);
    }
    __syncwarp();
  } else if ((MX || CG2) && warp == 2 + C::EPI_WARPS) {
    // ------------------------------------------------- scale-atom copier
    // Each stage's scale atoms go from shared memory to the stage's TMEM
    // columns once its data has landed; the commit tells the MMA thread.
    // A slot's columns are rewritten only after the producer refilled the
    // slot, i.e. after the MMAs that read them completed.  CTA pairs: the
    // MMA thread copies the atoms; this warp builds the SwiGLU weight atom
    // and reports each stage in place to rank 0 (both CTAs).
    uint32_t it = 0, gc = 0, cur = 0;   // scale-atom groups (SFG): next, and the current one
    bool ok = true;
    TileWalk<MODE> w;
    w.start(p, cid);
    for (; ok && w.tile < num_tiles; w.advance(p)) {
      const Tile t = tile_at(w);
      for (int ks = 0; ks < t.kstages; ++ks, ++it) {
        const uint32_t slot = it % S, ph = (it / S) & 1;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait<CG2>(&full[slot], ph, abort_flag, p.err))) {
          ok = false;
          break;
        }
        if (C::SFG && ks % C::GS == 0) {
          cur = gc++;
          if (!__all_sync(0xFFFFFFFFu,
                          mbar_wait(&sfg_full[cur % C::SFR], (cur / C::SFR) & 1, abort_flag, p.err))) {
            ok = false;
            break;
          }
        }
        if (MX && PAIR && EPI == kEpiSwigluFwd) {
          // The A tile is rows f0..f0+63 of the gate half, then of the up
          // half: its atom (row p at byte (p%32)*16 + (p/32)*4 + l) takes
          // rows 64a..64a+63 (a = (f0/64) % 2) of the gate half's 128-row
          // atom, then the same rows of the up half's.  Lane r builds its
          // 16 bytes from 8 of each, over the gate atom's place.
          // (CTA pairs: for each of the stage's two K-chunks; the up half's
          // atoms follow the gate half's)
          const int a8 = ((t.out_col0 >> 6) & 1) * 8;
#pragma unroll
          for (int c = 0; c < C::KCH; ++c) {
            uint8_t* at = smem + slot * C::STAGE + C::SF_OFF + c * kAtom;
            const uint2 g = *reinterpret_cast<const uint2*>(at + lane * 16 + a8);
            const uint2 u = *reinterpret_cast<const uint2*>(at + C::KCH * kAtom + lane * 16 + a8);
            __syncwarp();
            *reinterpret_cast<uint4*>(at + lane * 16) = make_uint4(g.x, g.y, u.x, u.y);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (CG2) {
          if (lane == 0) {
            if (rank == 0) mbar_arrive(&ready[slot]);
            else mbar_arrive_cluster(cluster_addr(&ready[slot], 0));
          }
          __syncwarp();
          continue;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sfcol = tmem + C::SF_COL0 + slot * C::SF_COLS;
          if (C::SFG) {
            const uint32_t grp = smem_u32(sfg + (cur % C::SFR) * C::GROUP_BYTES) + (ks % C::GS) * kAtom;
            tc_cp_sf(sfcol, sdesc_sf_atom(grp));
            tc_cp_sf(sfcol + 4, sdesc_sf_atom(grp + C::GS * kAtom));
            // the group's last stage: its buffer may be refilled once these copies completed
            if (ks % C::GS == C::GS - 1 || ks == t.kstages - 1) tc_commit(&sfg_empty[cur % C::SFR]);
          } else if (PAIR) {
            // the weight's atom (SwiGLU: built above), then the pair's B atoms
            const uint32_t ssf = smem_u32(smem + slot * C::STAGE) + C::SF_OFF;
            tc_cp_sf(sfcol, sdesc_sf_atom(ssf));
            tc_cp_sf(sfcol + 4, sdesc_sf_atom(ssf + 2 * kAtom));
            if (t.b_rows > 128) tc_cp_sf(sfcol + 8, sdesc_sf_atom(ssf + 3 * kAtom));
          } else {
            const uint32_t ssf = smem_u32(smem + slot * C::STAGE) + NA * kABytes + kBBytes;
#pragma unroll
            for (int j = 0; j <= NA; ++j) tc_cp_sf(sfcol + j * 4, sdesc_sf_atom(ssf + j * kAtom));
          }
          tc_commit(&sf_full[slot]);
        }
        __syncwarp();
      }
    }
    // every copy issued here must be complete before TMEM is released
    if (lane == 0 && !CG2) {
      tc_commit(sf_drain);
      drain_wait(sf_drain, 0);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue
    const int q = warp & 3;              // TMEM lane quadrant of this warp
    const int hw = (warp - 2) >> 2;      // 0 .. EPI_WARPS/4 - 1
    const int grp = hw / 2 % C::EPI_GROUPS;   // weight gradient: group of this warp
    const int h = C::EPI_GROUPS > 1 ? (hw & 1) : hw;  // which 32-column chunks it drains
    const int lrow = q * 32 + lane;
    const int gtid = (threadIdx.x - 64) % C::GROUP_THREADS;   // thread index within the group
    const bool staged = C::WGRAD && p.tma_store;
    uint32_t tc = grp;
    // (the epilogue has slack: it decodes each tile from its index, which
    // keeps the walk's registers out of its register-bound loop)
    for (int tile = cid + grp * ncl; tile < num_tiles; tile += C::EPI_GROUPS * ncl, tc += C::EPI_GROUPS) {
      TileWalk<MODE> w;
      w.start(p, tile);
      const Tile t = tile_at(w);
      const uint32_t acc = tc % C::ACC_BUFS, aph = (tc / C::ACC_BUFS) & 1;
      uint32_t hp[32];
      if (EPI == kEpiSwigluBwd && 32 * h < t.b_rows) load_h1_chunk(p, t, t.out_col0 + lrow, 32 * h, hp);
      const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait<CG2>(&tfull[acc], aph, abort_flag, p.err));
      constexpr bool pair_swiglu = PAIR && EPI == kEpiSwigluFwd;   // leaves through its own barrier
      if (!staged && !pair_swiglu && !ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * C::ACC_COLS;
      if (staged) {
        // The group's 8 warps drain the 128 x 128 accumulator into the
        // group's 32 KB staging buffer and its store thread (gtid 0) moves it
        // out with TMA.  The first TMEM read starts first; while it is in
        // flight the store thread makes sure its previous TMA store has
        // finished reading the buffer.  Every warp of the group reaches the
        // barrier once per tile whether its bounded wait succeeded or not, so
        // a warp that gives up cannot leave the others blocked in it: they
        // all see the group's flag and leave together.
        //  * BF16: two 64-column boxes, chunks 32h and 32h + 64 of each warp.
        //  * FP32 (store or reduce-add): two passes over 64 columns, each
        //    two 32-column boxes; in pass hh the warp drains chunk
        //    64 hh + 32 h into box h.  A reduce-add into an expert without
        //    rows is skipped (its dW stays as it was).
        uint8_t* stg = staging + grp * 32768;
        constexpr bool f32 = DWF;
        const bool has = ok && t.kstages > 0;
        uint32_t r[32];
        if (has) tmem_ld32(tbase + 32 * h, r);
        if (!ok && lane == 0) epi_abort[grp] = 1;
        if (gtid == 0) bulk_wait_read<0>();
        named_bar_sync(kEpiBarrier + grp, C::GROUP_THREADS);
        tmem_ld_wait();
        if (epi_abort[grp]) break;
        const int y = t.e * p.m_tiles * 128 + t.out_row0;
        if (!f32) {
          stage_chunk(r, !has, 32 * h, lrow, stg);
          if (has) {
            tmem_ld32(tbase + 32 * h + 64, r);
            tmem_ld_wait();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
          stage_chunk(r, !has, 32 * h + 64, lrow, stg);
          fence_proxy_async_smem();
          named_bar_sync(kEpiBarrier + grp, C::GROUP_THREADS);
          if (gtid == 0) {
            tma_store_2d(&tmC, stg, t.out_col0, y);
            tma_store_2d(&tmC, stg + 16384, t.out_col0 + 64, y);
            bulk_commit();
          }
          continue;
        }
        const bool add = p.tma_store == kDwAddF32;
        if (add && t.kstages == 0) {   // nothing to add: the group leaves the tile together
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
          continue;
        }
        stage_chunk_f32(r, !has, h, lrow, stg);
        fence_proxy_async_smem();
        named_bar_sync(kEpiBarrier + grp, C::GROUP_THREADS);
        if (gtid == 0) {
          for (int b = 0; b < 2; ++b) {
            if (add) tma_reduce_add_2d(&tmC, stg + b * 16384, t.out_col0 + 32 * b, y);
            else tma_store_2d(&tmC, stg + b * 16384, t.out_col0 + 32 * b, y);
          }
          bulk_commit();
        }
        // the second half: its TMEM read overlaps the first half's store
        if (has) tmem_ld32(tbase + 64 + 32 * h, r);
        if (gtid == 0) bulk_wait_read<0>();   // the second half reuses the buffer
        named_bar_sync(kEpiBarrier + grp, C::GROUP_THREADS);
        if (has) tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        stage_chunk_f32(r, !has, h, lrow, stg);
        fence_proxy_async_smem();
        named_bar_sync(kEpiBarrier + grp, C::GROUP_THREADS);
        if (gtid == 0) {
          for (int b = 0; b < 2; ++b) {
            if (add) tma_reduce_add_2d(&tmC, stg + b * 16384, t.out_col0 + 64 + 32 * b, y);
            else tma_store_2d(&tmC, stg + b * 16384, t.out_col0 + 64 + 32 * b, y);
          }
          bulk_commit();
        }
        continue;
      }
      if (EPI == kEpiStore) epi_store<NA, PAIR ? 4 : 2>(p, t, tbase, lrow, lane, h, &tempty[acc]);
      else if (pair_swiglu) {
        if (!epi_swiglu_fwd_pair<MX>(p, t, tbase, q, lane, h, ok, &tempty[acc], xbuf, epi_abort, kEpiBarrier,
                                     C::EPI_THREADS))
          break;
      } else if (EPI == kEpiSwigluFwd) epi_swiglu_fwd<MX>(p, t, tbase, lrow, lane, h, &tempty[acc]);
      else if (EPI == kEpiSwigluBwd) {
        // its two accumulator buffers cover this (heavier) epilogue: release at the end
        epi_swiglu_bwd<MX>(p, t, tbase, lrow, lane, h, hp);
        release_acc(&tempty[acc], lane);
      } else {
        epi_wgrad_direct(p, t, tbase, q, lane, h, 64,
                         reinterpret_cast<float*>(staging + grp * 32768 + (gtid >> 5) * 4096));
        release_acc(&tempty[acc], lane);
      }
    }
    if (staged && gtid == 0) bulk_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  // CTA pairs: neither CTA leaves (nor frees TMEM) while the other may still
  // touch its shared memory, barriers or tensor memory
  if (CG2) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_cg<CG>(tmem, 512);
  }
}

template <bool MX, int NA, int EPI, int MODE, bool DWF = false>
cudaError_t launch_impl(const GemmLaunch& g, int num_sms, cudaStream_t stream) {
  using C = Cfg<MX, NA, MODE>;
  auto kern = gemm_kernel<MX, NA, EPI, MODE, DWF>;
  static PerDeviceOnce setup;
  static int pair_slots[kMaxDevices];   // CTA pairs: clusters of two that fit on the device at once
  int dev = 0;
  cudaError_t se = cudaGetDevice(&dev);
  if (se != cudaSuccess) return se;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute la[1];
  la[0].id = cudaLaunchAttributeClusterDimension;
  la[0].val.clusterDim.x = 2;
  la[0].val.clusterDim.y = 1;
  la[0].val.clusterDim.z = 1;
  lc.blockDim = dim3(C::THREADS);
  lc.dynamicSmemBytes = C::SMEM;
  lc.stream = stream;
  lc.attrs = la;
  lc.numAttrs = 1;
  se = setup.once([&] {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess || !C::CG2) return e;
    int n = 0;
    lc.gridDim = dim3(2);
    e = cudaOccupancyMaxActiveClusters(&n, kern, &lc);
    if (e == cudaSuccess && n < 1) e = cudaErrorInvalidConfiguration;
    pair_slots[dev] = n;
    return e;
  });
  if (se != cudaSuccess) return se;
  // CTA pairs: the walk is over clusters (both CTAs of one take the same tiles)
  const int units = C::CG2 ? max(1, min(min(num_sms / 2, pair_slots[dev]), g.max_tiles))
                           : max(1, min(num_sms, g.max_tiles));
  GemmParams p = g.p;
  const int q = units / p.n_tiles;
  p.walk[0] = units;
  p.walk[1] = units % p.n_tiles;
  p.walk[2] = MODE != kGroupedK ? q : q % p.m_tiles;
  p.walk[3] = MODE != kGroupedK ? 0 : q / p.m_tiles;
  if (C::CG2) {
    lc.gridDim = dim3(2 * units);
    return cudaLaunchKernelEx(&lc, kern, g.tmA, g.tmB, g.tmC, g.aux[0], g.aux[1], g.aux[2], g.aux[3], p);
  }
  kern<<<units, C::THREADS, C::SMEM, stream>>>(g.tmA, g.tmB, g.tmC, g.aux[0], g.aux[1], g.aux[2], g.aux[3], p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(const GemmLaunch& g, int num_sms, cudaStream_t stream) {
  if (g.max_tiles <= 0) return cudaSuccess;
  // B boxes must tile every row block (32-row multiples) or the 128-row K-mode tile
  if (g.p.b_box_rows != 32 && !(g.p.b_box_rows == 128 && g.mode == kGroupedK)) return cudaErrorInvalidValue;
#define MOE_GEMM_CASE(MXV, NAV, EPIV, MODEV)                                         \
  if (g.mx == MXV && g.na == NAV && g.epi == EPIV && g.mode == MODEV)                \
    return launch_impl<MXV, NAV, EPIV, MODEV>(g, num_sms, stream);
  MOE_GEMM_CASE(false, 2, kEpiSwigluFwd, kGroupedM)
  MOE_GEMM_CASE(true, 2, kEpiSwigluFwd, kGroupedM)
  MOE_GEMM_CASE(false, 1, kEpiStore, kGroupedM)
  MOE_GEMM_CASE(true, 1, kEpiStore, kGroupedM)
  MOE_GEMM_CASE(false, 2, kEpiStore, kGroupedM)
  MOE_GEMM_CASE(true, 2, kEpiStore, kGroupedM)
  MOE_GEMM_CASE(false, 1, kEpiSwigluBwd, kGroupedM)
  MOE_GEMM_CASE(true, 1, kEpiSwigluBwd, kGroupedM)
  MOE_GEMM_CASE(false, 1, kEpiSwigluFwd, kGroupedMP)
  MOE_GEMM_CASE(true, 1, kEpiSwigluFwd, kGroupedMP)
  MOE_GEMM_CASE(false, 1, kEpiStore, kGroupedMP)
  MOE_GEMM_CASE(false, 1, kEpiSwigluBwd, kGroupedMP)
  MOE_GEMM_CASE(true, 1, kEpiStore, kGroupedMP)
  MOE_GEMM_CASE(false, 1, kEpiSwigluFwd, kGroupedMC)
  MOE_GEMM_CASE(true, 1, kEpiSwigluFwd, kGroupedMC)
  MOE_GEMM_CASE(false, 1, kEpiStore, kGroupedMC)
  MOE_GEMM_CASE(true, 1, kEpiStore, kGroupedMC)
  MOE_GEMM_CASE(false, 1, kEpiSwigluBwd, kGroupedMC)
  if (g.epi == kEpiWgrad && g.mode == kGroupedK &&
      (g.p.tma_store == kDwStoreF32 || g.p.tma_store == kDwAddF32))
    return g.mx ? launch_impl<true, 1, kEpiWgrad, kGroupedK, true>(g, num_sms, stream)
                : launch_impl<false, 1, kEpiWgrad, kGroupedK, true>(g, num_sms, stream);
  MOE_GEMM_CASE(false, 1, kEpiWgrad, kGroupedK)
  MOE_GEMM_CASE(true, 1, kEpiWgrad, kGroupedK)
#undef MOE_GEMM_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe
