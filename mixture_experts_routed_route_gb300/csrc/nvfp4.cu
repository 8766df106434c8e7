// NVFP4 inference: weight preparation, row quantisation and the grouped
// GEMMs of the routed forward.
//
// Format ("Dist-MoE: Speed-of-light distributed Mixture-of-Experts
// kernels", section 02, "Expert Computation and Tensor Precision": E2M1
// values packed two per byte, E4M3 block scales and a global scale per row;
// section 08, "Public API and Supported Modes": NVFP4 inference with
// prepared weights).  Along the contraction axis K: blocks of 16 values,
// one E4M3 block scale each, one FP32 global scale g per row, every
// quantiser step one FP32 operation (round to nearest even) in this order:
//     g = a_row / 2688, s6g = 6 g, sb = E4M3(a_block / s6g), d = sb g,
//     q = E2M1(v / d)      (q = 0 where d = 0),
// and v is represented by q * sb * g.  E4M3 and E2M1 saturate (448, 6).
//
// Layout: "chunks" of 128 rows x 64 values, one GEMM stage each: 4096 bytes
// of codes (row m at byte 32 m; value k of the row in byte k / 2, the low
// nibble for even k), then 512 bytes of block scales (row m's four at
// 4096 + 4 m).
//   Weights [E, N, K]: the chunk of row tile t = (e N + n) / 128 and stage s
//   at (t * K / 64 + s) * 4608; g [E * N] FP32.
//   Routed activations: the chunk of routing block b and stage s at
//   (b * K / 64 + s) * 4608, the block's row p at the chunk's row p (rows
//   past the block are never written and never read); g [r_cap] per row.
//
// GEMM.  q * sb is exact in FP16 (a 2-bit E2M1 significand times a 4-bit
// E4M3 one, magnitudes 2^-10 .. 2688), so the kernel does not need the
// tensor cores' own FP4 form: expander warps turn each stage's codes and
// block scales into FP16 tiles in shared memory (the 128-byte-swizzled
// K-major layout TMA would write), the documented kind::f16 MMA (A = B =
// FP16) accumulates sum_k q_a sb_a q_b sb_b in FP32 in TMEM, and the
// epilogue multiplies by g_a g_b.  HBM carries 4.5 bits per weight value.
// Warp roles (448 threads): 0 copies chunks into a staging ring (bulk
// copies, one per operand per stage); 1 issues the MMAs and owns TMEM; 2-5
// drain the double-buffered accumulator; 6-13 expand.  Tiles: routing
// block m x 128 output features (the SwiGLU GEMM takes 128 gate and the
// 128 matching up rows as two A tiles with two accumulators), walked
// block by block like the other grouped-M GEMMs.
#include <cuda_fp16.h>

#include "gemm_core.cuh"   // drain_wait

namespace moe {

namespace {

constexpr int kF4Codes = 128 * 32;            // code bytes of a chunk
constexpr int kF4Chunk = kF4Codes + 128 * 4;  // + 4 block scales per row
constexpr int kF4Tile = 128 * 128;            // an FP16 operand tile: 128 rows x 64 values
constexpr float kF4GlobalDiv = 2688.0f;       // largest E2M1 (6) x largest E4M3 (448)

// ------------------------------------------------------------ conversions

// Value of an E4M3 code (low byte), exact through FP16.
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(code & 0xFFu)));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// Two floats -> two E2M1 codes (lo in bits 0-3), nearest even, saturating.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 b;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b, %2, %1;\n\t"
      "mov.b16 %0, {b, 0};\n\t}"
      : "=h"(r)
      : "f"(lo), "f"(hi));
  return r;
}

// Four code bytes (8 values) -> four FP16 pairs, in value order.
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
      "mov.b32 {c0, c1, c2, c3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, c0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, c1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, c2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, c3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// One block of 16 values: returns its E4M3 scale code and writes its 8 code
// bytes (values 0-7 in w.x, 8-15 in w.y).
__device__ __forceinline__ uint32_t quantise_block(const float (&v)[16], float g, float s6g, uint2& w) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(v[i]));
  const float ratio = s6g > 0.0f ? __fdiv_rn(a, s6g) : 0.0f;
  const uint32_t sbc = cvt_e4m3x2(ratio, 0.0f) & 0xFFu;
  const float d = __fmul_rn(e4m3_value(sbc), g);
  uint32_t c[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float y0 = d > 0.0f ? __fdiv_rn(v[2 * i], d) : 0.0f;
    const float y1 = d > 0.0f ? __fdiv_rn(v[2 * i + 1], d) : 0.0f;
    c[i >> 2] |= cvt_e2m1x2(y0, y1) << (8 * (i & 3));
  }
  w = make_uint2(c[0], c[1]);
  return sbc;
}

// 16 consecutive values of a row as FP32 (BF16 or FP32 source; zeros when
// the row is absent).
template <bool F32>
__device__ __forceinline__ void load16(const void* row, int k0, float (&v)[16]) {
  if (!row) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.0f;
    return;
  }
  if (F32) {
    const float4* s = reinterpret_cast<const float4*>(static_cast<const float*>(row) + k0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 f = s[q];
      v[4 * q] = f.x;
      v[4 * q + 1] = f.y;
      v[4 * q + 2] = f.z;
      v[4 * q + 3] = f.w;
    }
  } else {
    const uint4* s = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(row) + k0);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint4 u = __ldg(s + q);
      const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * q + 2 * j] = bf16_lo(ww[j]);
        v[8 * q + 2 * j + 1] = bf16_hi(ww[j]);
      }
    }
  }
}

// ------------------------------------------------------- row quantisation
// One warp per row.  SRC 0: weight rows (BF16 [rows, K], row i in chunk
// row tile i / 128); 1: routed x rows (BF16 x[perm[r] / top_k], zeros for a
// pad row); 2: routed FP32 rows (h2 [r_cap, K]).  Pass 1 takes the row's
// maximum magnitude, pass 2 re-reads the row (from L1/L2) block by block:
// lane l takes blocks l, l + 32, ...; the four lanes of one stage's blocks
// gather their scale bytes into one word.
template <int SRC>
__global__ void __launch_bounds__(256) nvfp4_rows_kernel(const void* __restrict__ src, int K, int top_k,
                                                         int nrows_host, const int* __restrict__ hdr,
                                                         const int* __restrict__ perm,
                                                         const int* __restrict__ row_block,
                                                         const int4* __restrict__ blocks, uint8_t* __restrict__ chunks,
                                                         float* __restrict__ g_out) {
  constexpr bool F32 = SRC == 2;
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int rows = SRC == 0 ? nrows_host : hdr[2];
  const int ks = K / 64, nb = K / 16;
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    const void* row = nullptr;
    uint8_t* base;
    int p;
    if (SRC == 0) {
      row = static_cast<const __nv_bfloat16*>(src) + static_cast<long long>(r) * K;
      base = chunks + static_cast<long long>(r >> 7) * ks * kF4Chunk;
      p = r & 127;
    } else {
      if (SRC == 1) {
        const int route = perm[r];
        if (route >= 0) row = static_cast<const __nv_bfloat16*>(src) + static_cast<long long>(route / top_k) * K;
      } else {
        row = static_cast<const float*>(src) + static_cast<long long>(r) * K;
      }
      const int b = row_block[r >> 5];
      base = chunks + static_cast<long long>(b) * ks * kF4Chunk;
      p = r - blocks[b].y;
    }
    float a = 0.0f;
    if (row) {
      for (int k0 = 16 * lane; k0 < K; k0 += 512) {
        float v[16];
        load16<F32>(row, k0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(v[i]));
      }
    }
    a = warp_max_nonneg(a);
    const float g = __fdiv_rn(a, kF4GlobalDiv);
    const float s6g = __fmul_rn(6.0f, g);
    for (int kb0 = 0; kb0 < nb; kb0 += 32) {
      const int kb = kb0 + lane;
      const bool act = kb < nb;   // nb is a multiple of 8: a stage's four lanes agree
      uint2 w = make_uint2(0u, 0u);
      uint32_t sbc = 0;
      if (act) {
        float v[16];
        load16<F32>(row, 16 * kb, v);
        sbc = quantise_block(v, g, s6g, w);
      }
      uint32_t sw = sbc << (8 * (lane & 3));
      sw |= __shfl_xor_sync(0xFFFFFFFFu, sw, 1);
      sw |= __shfl_xor_sync(0xFFFFFFFFu, sw, 2);
      if (act) {
        uint8_t* ch = base + static_cast<long long>(kb >> 2) * kF4Chunk;
        *reinterpret_cast<uint2*>(ch + p * 32 + (kb & 3) * 8) = w;
        if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(ch + kF4Codes + p * 4) = sw;
      }
    }
    if (lane == 0) g_out[r] = g;
  }
}

// ------------------------------------------------------------------- GEMM

constexpr int kF4Producer = 0, kF4Mma = 1, kF4Exp0 = 6, kF4ExpWarps = 8;   // warps 2-5: epilogue
constexpr int kF4Threads = (kF4Exp0 + kF4ExpWarps) * 32;   // 448

// NA A tiles per stage (2: the SwiGLU GEMM's gate and up tiles) and one B
// tile.  Staging slots hold chunks as copied; operand slots hold the FP16
// tiles the MMAs read.  One accumulator buffer is NA x 128 columns, two
// buffers alternate.
template <int NA>
struct F4Cfg {
  static constexpr int STG = NA == 2 ? 5 : 8;
  static constexpr int OPS = NA == 2 ? 3 : 4;
  static constexpr int STG_BYTES = (NA + 1) * kF4Chunk;
  static constexpr int OP_BYTES = (NA + 1) * kF4Tile;
  static constexpr int ACC_COLS = NA * 128;
  static constexpr int TMEM_COLS = 2 * ACC_COLS;
  static constexpr int SMEM = 1024 + OPS * OP_BYTES + STG * STG_BYTES + 256;
};

// Row m, values 32 h .. 32 h + 31 of a chunk: 16 code bytes and two block
// scales.  The expanders load every operand's row half before they store
// any tile (the stores could otherwise alias the next load, which would
// then wait for them).
struct RowHalf {
  uint4 codes;
  uint16_t scales;
};

__device__ __forceinline__ RowHalf load_row_half(const uint8_t* ch, int m, int h) {
  RowHalf r;
  r.codes = *reinterpret_cast<const uint4*>(ch + m * 32 + h * 16);
  r.scales = *reinterpret_cast<const uint16_t*>(ch + kF4Codes + m * 4 + h * 2);
  return r;
}

// Expand a row half into an FP16 tile: the tile's 16-byte chunk c of row m
// lies at m * 128 + ((c ^ (m % 8)) << 4).  q * sb is exact in FP16.
__device__ __forceinline__ void store_row_half(const RowHalf& rh, uint8_t* tile, int m, int h) {
  const uint4 cw = rh.codes;
  uint32_t s2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2) : "h"(rh.scales));
  const uint32_t s_lo = __byte_perm(s2, 0u, 0x1010), s_hi = __byte_perm(s2, 0u, 0x3232);
  const uint32_t ww[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t f[4];
    e2m1x8_to_f16(ww[j], f);
    const uint32_t s = j < 2 ? s_lo : s_hi;   // block 2h covers words 0-1, block 2h + 1 words 2-3
    const int c = 4 * h + j;
    *reinterpret_cast<uint4*>(tile + m * 128 + ((c ^ (m & 7)) << 4)) =
        make_uint4(hmul2(f[0], s), hmul2(f[1], s), hmul2(f[2], s), hmul2(f[3], s));
  }
}

template <int NA>
__global__ void __launch_bounds__(kF4Threads, 1) nvfp4_gemm_kernel(const Fp4GemmParams p) {
  using C = F4Cfg<NA>;
  extern __shared__ uint8_t f4_smem_raw[];
  uint8_t* ops = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(f4_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stg = ops + C::OPS * C::OP_BYTES;
  uint64_t* sfull = reinterpret_cast<uint64_t*>(stg + C::STG * C::STG_BYTES);   // chunks landed
  uint64_t* sempty = sfull + C::STG;    // chunks expanded (every expander thread)
  uint64_t* ofull = sempty + C::STG;    // FP16 tiles written (every expander thread)
  uint64_t* oempty = ofull + C::OPS;    // the MMAs reading them completed
  uint64_t* tfull = oempty + C::OPS;    // [2] accumulator complete
  uint64_t* tempty = tfull + 2;         // [2] accumulator drained (epilogue warps)
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STG; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], kF4ExpWarps * 32);
    }
    for (int o = 0; o < C::OPS; ++o) {
      mbar_init(&ofull[o], kF4ExpWarps * 32);
      mbar_init(&oempty[o], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kF4Mma) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int num_tiles = p.hdr[1] * p.n_tiles;

  if (warp == kF4Producer) {
    // ------------------------------------------------------ chunk copies
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
      const int m = tile / p.n_tiles, n = tile - m * p.n_tiles;
      const int e = p.blocks[m].x;
      const uint8_t* a0 = p.a + static_cast<long long>(e * p.a_tiles_e + n) * p.ks * kF4Chunk;
      const uint8_t* a1 = p.a + static_cast<long long>(e * p.a_tiles_e + p.n_tiles + n) * p.ks * kF4Chunk;
      const uint8_t* b0 = p.b + static_cast<long long>(m) * p.ks * kF4Chunk;
      for (int s = 0; s < p.ks; ++s, ++it) {
        const uint32_t slot = it % C::STG, ph = (it / C::STG) & 1;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sempty[slot], ph ^ 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* st = stg + slot * C::STG_BYTES;
          const long long off = static_cast<long long>(s) * kF4Chunk;
          mbar_arrive_expect_tx(&sfull[slot], C::STG_BYTES);
          bulk_load(st, a0 + off, kF4Chunk, &sfull[slot]);
          if (NA == 2) bulk_load(st + kF4Chunk, a1 + off, kF4Chunk, &sfull[slot]);
          bulk_load(st + NA * kF4Chunk, b0 + off, kF4Chunk, &sfull[slot]);
        }
        __syncwarp();
      }
    }
    // no copy may still be landing in shared memory when the CTA exits
    if (lane == 0) {
      const uint32_t pend = it < static_cast<uint32_t>(C::STG) ? it : static_cast<uint32_t>(C::STG);
      for (uint32_t j = 0; j < pend; ++j) {
        const uint32_t i2 = it - 1 - j;
        drain_wait(&sfull[i2 % C::STG], (i2 / C::STG) & 1);
      }
    }
    __syncwarp();
  } else if (warp >= kF4Exp0) {
    // ------------------------------------------------------- expanders
    // Thread x expands row x % 128, half x / 128 of every operand of the
    // stage (B only for the block's rows), makes its generic-proxy writes
    // visible to the async proxy and arrives on both barriers (measured
    // faster than one arrival per warp after a warp synchronisation).
    const int x = threadIdx.x - kF4Exp0 * 32;
    const int row = x & 127, h = x >> 7;
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
      const int nrows = p.blocks[tile / p.n_tiles].z;
      for (int s = 0; s < p.ks; ++s, ++it) {
        const uint32_t sl = it % C::STG, sph = (it / C::STG) & 1;
        const uint32_t ol = it % C::OPS, oph = (it / C::OPS) & 1;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sfull[sl], sph, abort_flag, p.err))) {
          ok = false;
          break;
        }
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&oempty[ol], oph ^ 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        const uint8_t* st = stg + sl * C::STG_BYTES;
        uint8_t* op = ops + ol * C::OP_BYTES;
        const bool brow = row < nrows;
        RowHalf rh[NA + 1];
#pragma unroll
        for (int u = 0; u < NA; ++u) rh[u] = load_row_half(st + u * kF4Chunk, row, h);
        if (brow) rh[NA] = load_row_half(st + NA * kF4Chunk, row, h);
#pragma unroll
        for (int u = 0; u < NA; ++u) store_row_half(rh[u], op + u * kF4Tile, row, h);
        if (brow) store_row_half(rh[NA], op + NA * kF4Tile, row, h);
        fence_proxy_async_smem();
        mbar_arrive(&sempty[sl]);
        mbar_arrive(&ofull[ol]);
      }
    }
  } else if (warp == kF4Mma) {
    // ------------------------------------------------------------ MMAs
    uint32_t it = 0, tc = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++tc) {
      const int nrows = p.blocks[tile / p.n_tiles].z;
      const uint32_t acc = tc & 1, aph = (tc >> 1) & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tempty[acc], aph ^ 1, abort_flag, p.err))) break;
      tc_fence_after();
      // kind::f16: D = F32 (bits 4-5 = 1), A = B = F16 (format 0 at bits
      // 7-9 and 10-12), both K-major, N >> 3 at bits 17-22, M = 128 (M >> 4
      // at bits 24-28); N = the block's rows (a multiple of 32)
      const uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(nrows >> 3) << 17) | ((128u >> 4) << 24);
      const uint32_t d0 = tmem + acc * C::ACC_COLS;
      for (int s = 0; s < p.ks; ++s, ++it) {
        const uint32_t ol = it % C::OPS, oph = (it / C::OPS) & 1;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&ofull[ol], oph, abort_flag, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = smem_u32(ops + ol * C::OP_BYTES);
          const uint64_t bd = sdesc_k_sw128(sa + NA * kF4Tile);
#pragma unroll
          for (int k = 0; k < 4; ++k) {   // 16 FP16 values (32 bytes) of K each
#pragma unroll
            for (int j = 0; j < NA; ++j)
              mma_bf16(d0 + j * 128, sdesc_k_sw128(sa + j * kF4Tile) + 2 * k, bd + 2 * k, idesc,
                       (s | k) ? 1u : 0u);
          }
          tc_commit(&oempty[ol]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc_commit(&tfull[acc]);
      __syncwarp();
    }
    // every MMA issued here must be complete before TMEM is released
    if (lane == 0) {
      tc_commit(drain);
      drain_wait(drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- epilogue
    // Warp w drains TMEM lanes 32 (w % 4) ..: output features n * 128 +
    // 32 (w % 4) + lane, 32 token columns per read.  SwiGLU: g and u =
    // BF16(acc * g_a * g_b), h2 = SiLU(g) * u in FP32 (clamped first when a
    // limit is set) to the FP32 h2 rows; otherwise h3 = BF16(acc g_a g_b).
    const int q = warp & 3;
    const int lrow = 32 * q + lane;
    const float L = p.swiglu_limit;
    uint32_t tc = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tc) {
      const int m = tile / p.n_tiles, n = tile - m * p.n_tiles;
      const int4 blk = p.blocks[m];
      const uint32_t acc = tc & 1, aph = (tc >> 1) & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tfull[acc], aph, abort_flag, p.err))) break;
      tc_fence_after();
      const int f = n * 128 + lrow;
      const float ga0 = p.ga[static_cast<long long>(blk.x * p.a_tiles_e + n) * 128 + lrow];
      const float ga1 = NA == 2 ? p.ga[static_cast<long long>(blk.x * p.a_tiles_e + p.n_tiles + n) * 128 + lrow] : 0.0f;
      const uint32_t tb = tmem + (static_cast<uint32_t>(32 * q) << 16) + acc * C::ACC_COLS;
      int cg = 0, cu = 0;
      for (int c0 = 0; c0 < blk.z; c0 += 32) {
        uint32_t r0[32], r1[32];
        tmem_ld32(tb + c0, r0);
        if (NA == 2) tmem_ld32(tb + 128 + c0, r1);
        tmem_ld_wait();
        const float gbl = p.gb[blk.y + c0 + lane];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float gb = __shfl_sync(0xFFFFFFFFu, gbl, j);
          const long long r = blk.y + c0 + j;
          if (NA == 2) {
            float g = bf16_round(__uint_as_float(r0[j]) * ga0 * gb);
            float u = bf16_round(__uint_as_float(r1[j]) * ga1 * gb);
            if (L > 0.0f) {
              cg += g > L;
              cu += fabsf(u) > L;
              g = fminf(g, L);
              u = fminf(fmaxf(u, -L), L);
            }
            static_cast<float*>(p.out)[r * p.ld + f] = silu_f(g) * u;
          } else {
            static_cast<__nv_bfloat16*>(p.out)[r * p.ld + f] =
                __float2bfloat16_rn(__uint_as_float(r0[j]) * ga0 * gb);
          }
        }
      }
      if (NA == 2 && L > 0.0f && p.clip != nullptr) {
        cg = __reduce_add_sync(0xFFFFFFFFu, cg);
        cu = __reduce_add_sync(0xFFFFFFFFu, cu);
        if (lane == 0) {
          if (cg) atomicAdd(&p.clip[0], static_cast<unsigned long long>(cg));
          if (cu) atomicAdd(&p.clip[1], static_cast<unsigned long long>(cu));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kF4Mma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int NA>
cudaError_t gemm_impl(const Fp4GemmParams& p, int grid, cudaStream_t stream) {
  using C = F4Cfg<NA>;
  auto kern = nvfp4_gemm_kernel<NA>;
  static PerDeviceOnce setup;
  const cudaError_t se =
      setup.once([&] { return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM); });
  if (se != cudaSuccess) return se;
  kern<<<grid, kF4Threads, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

template <int SRC>
cudaError_t rows_impl(const void* src, int K, int top_k, int rows, const RoutingPtrs* rp, uint8_t* chunks, float* g,
                      int num_sms, cudaStream_t stream) {
  const int blocks = max(1, min((rows + 7) / 8, num_sms * 8));
  nvfp4_rows_kernel<SRC><<<blocks, 256, 0, stream>>>(src, K, top_k, rows, rp ? rp->hdr : nullptr,
                                                     rp ? rp->perm : nullptr, rp ? rp->row_block : nullptr,
                                                     rp ? rp->blocks : nullptr, chunks, g);
  return cudaGetLastError();
}

}  // namespace

size_t nvfp4_chunk_bytes(long long row_tiles, int K) {
  return static_cast<size_t>(row_tiles) * static_cast<size_t>(K / 64) * kF4Chunk;
}

cudaError_t launch_nvfp4_prep_weight(const void* w, int E, int N, int K, uint8_t* chunks, float* g, int num_sms,
                                     cudaStream_t stream) {
  return rows_impl<0>(w, K, 1, E * N, nullptr, chunks, g, num_sms, stream);
}

cudaError_t launch_nvfp4_rows(bool f32_rows, const void* src, int K, int top_k, const RoutingPtrs& rp, int r_cap,
                              uint8_t* chunks, float* g, int num_sms, cudaStream_t stream) {
  return f32_rows ? rows_impl<2>(src, K, top_k, r_cap, &rp, chunks, g, num_sms, stream)
                  : rows_impl<1>(src, K, top_k, r_cap, &rp, chunks, g, num_sms, stream);
}

cudaError_t launch_nvfp4_gemm(const Fp4GemmParams& p, bool swiglu, int grid, cudaStream_t stream) {
  return swiglu ? gemm_impl<2>(p, grid, stream) : gemm_impl<1>(p, grid, stream);
}

}  // namespace moe
