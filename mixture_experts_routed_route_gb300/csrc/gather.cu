// F1 / B0: gather token rows into expert-major order, optionally scaled by
// the route's score, as BF16 or as MXFP8 (E4M3 + one E8M0 scale per 32
// values).
//
// Dist-MoE explainer section 02, "Quantization Axes for Forward and
// Backward": FPROP/DGRAD operands are scaled along the feature axis (row
// bundles, launch_gather_rows); WGRAD contracts over token rows and needs a
// separately quantised column-oriented bundle (stored transposed [D, r_cap]
// so the GEMM reads it K-major); launch_gather_both writes both bundles of
// the same rows in one pass when training.  In MXFP8 training the rows
// travel as BF16 and are quantised where they land (same section); row
// quantisation depends only on the row, so quantising after the gather is
// exact.  Pad rows (route -1) are zero.
//
// The dh3 prep of the backward ("Mixture of Experts: How Routing Becomes GPU
// Computation", section 2, "SwiGLU backward: the complete expert path":
// dH = p * dY) is the same gather with use_scores: the FP32 product of the
// score and the BF16 dY is what gets rounded or quantised.
#include "kernels.cuh"

namespace moe {

namespace {

__device__ __forceinline__ void unpack8(const uint4 u, float (&v)[8]) {
  v[0] = bf16_lo(u.x);
  v[1] = bf16_hi(u.x);
  v[2] = bf16_lo(u.y);
  v[3] = bf16_hi(u.y);
  v[4] = bf16_lo(u.z);
  v[5] = bf16_hi(u.z);
  v[6] = bf16_lo(u.w);
  v[7] = bf16_hi(u.w);
}

// One warp per row; each lane moves 8 values (16 bytes) per step, 4 lanes
// cover one 32-value MX block.
template <bool MX, bool SCALE>
__global__ void __launch_bounds__(256) gather_rows_kernel(const __nv_bfloat16* __restrict__ src, int D, int K,
                                                          const int* __restrict__ hdr, const int* __restrict__ perm,
                                                          const float* __restrict__ scores, void* __restrict__ dst,
                                                          uint8_t* __restrict__ dst_sf,
                                                          const int* __restrict__ row_block,
                                                          const int4* __restrict__ blocks) {
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int rows = hdr[2];
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    const int route = perm[r];
    const __nv_bfloat16* srow = nullptr;
    float s = 1.0f;
    // scale atoms of this row: routing block b, row p within it
    long long atom_row = 0;
    int p = 0;
    if (MX) {
      const int b = row_block[r >> 5];
      p = r - blocks[b].y;
      atom_row = static_cast<long long>(b) * (D / 128);
    }
    if (route >= 0) {
      srow = src + static_cast<long long>(route / K) * D;
      if (SCALE) s = scores[route];
    }
    // four 16-byte loads in flight per lane before any is used
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
      const bool act = c < D;
      uint4 u = ub[q];
      if (!MX) {
        if (SCALE) {
          float v[8];
          unpack8(u, v);
          u.x = pack_bf16x2(s * v[0], s * v[1]);
          u.y = pack_bf16x2(s * v[2], s * v[3]);
          u.z = pack_bf16x2(s * v[4], s * v[5]);
          u.w = pack_bf16x2(s * v[6], s * v[7]);
        }
        if (act) *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dst) + static_cast<long long>(r) * D + c) = u;
      } else {
        float v[8];
        unpack8(u, v);
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (SCALE) v[j] = s * v[j];
          amax = fmaxf(amax, fabsf(v[j]));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        const int e = mx_shared_exp(amax);
        const float inv = exp2_int(-e);
        uint2 q;
        q.x = cvt_e4m3x2(v[0] * inv, v[1] * inv) | (cvt_e4m3x2(v[2] * inv, v[3] * inv) << 16);
        q.y = cvt_e4m3x2(v[4] * inv, v[5] * inv) | (cvt_e4m3x2(v[6] * inv, v[7] * inv) << 16);
        if (act) {
          *reinterpret_cast<uint2*>(static_cast<uint8_t*>(dst) + static_cast<long long>(r) * D + c) = q;
          if ((lane & 3) == 0) {
            const int kb = c >> 5;
            dst_sf[(atom_row + (kb >> 2)) * 512 + sf_atom_byte(p, kb & 3)] = static_cast<uint8_t>(e + 127);
          }
        }
      }
      }
    }
  }
}

// Both bundles in one pass (training), BF16.  One CTA per (128-row tile,
// 128-column slab): the gathered rows go through shared memory once, then
//  * row bundle: warp w writes rows 16w .. 16w+15, lane l columns 4l .. 4l+3;
//  * column bundle: thread (c, half) writes feature c0+c for rows
//    64*half .. +63 (128 contiguous bytes per thread).
constexpr int kBothRows = 128, kBothCols = 128, kBothPitch = kBothCols + 4;
constexpr int kBothSmem = kBothRows * kBothPitch * 4;

template <bool SCALE>
__global__ void __launch_bounds__(256) gather_both_kernel(const __nv_bfloat16* __restrict__ src, int D, int K,
                                                          const int* __restrict__ hdr, const int* __restrict__ perm,
                                                          const float* __restrict__ scores,
                                                          __nv_bfloat16* __restrict__ dst,
                                                          __nv_bfloat16* __restrict__ dstT, int r_cap) {
  extern __shared__ float4 smem_f4[];
  float* tile = reinterpret_cast<float*>(smem_f4);  // [128][kBothPitch]
  const int rows = hdr[2];
  const int r0 = blockIdx.y * kBothRows;
  if (r0 >= rows) return;
  const int c0 = blockIdx.x * kBothCols;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // ---- load 128 gathered rows x 128 columns (16 chunks of 8 values per row):
  // thread t moves chunk t%16 of rows t/16 + 16j, j = 0..7.  All route
  // lookups are issued first, then all eight row loads, so a thread waits for
  // two memory latencies, not sixteen.
  {
    constexpr int kPer = kBothRows * 16 / 256;
    const int chunk = tid & 15, c = c0 + chunk * 8;
    int route[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int r = r0 + (tid >> 4) + 16 * j;
      route[j] = (r < r_cap) ? perm[r] : -1;
    }
    uint4 u[kPer];
    float s[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      u[j] = make_uint4(0, 0, 0, 0);
      s[j] = 1.0f;
      if (route[j] >= 0 && c < D) {
        u[j] = __ldg(reinterpret_cast<const uint4*>(src + static_cast<long long>(route[j] / K) * D + c));
        if (SCALE) s[j] = scores[route[j]];
      }
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      float v[8];
      unpack8(u[j], v);
      if (SCALE) {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = s[j] * v[q];
      }
      float4* t4 = reinterpret_cast<float4*>(tile + ((tid >> 4) + 16 * j) * kBothPitch + chunk * 8);
      t4[0] = make_float4(v[0], v[1], v[2], v[3]);
      t4[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
  __syncthreads();
  // ---- row bundle
  const int c = c0 + lane * 4;
  for (int rr = 0; rr < 16; ++rr) {
    const int row = warp * 16 + rr;
    const int r = r0 + row;
    const float4 x4 = *reinterpret_cast<const float4*>(tile + row * kBothPitch + lane * 4);
    if (c < D && r < rows)
      *reinterpret_cast<uint2*>(dst + static_cast<long long>(r) * D + c) =
          make_uint2(pack_bf16x2(x4.x, x4.y), pack_bf16x2(x4.z, x4.w));
  }
  // ---- column bundle
  const int cc = tid & 127, half = tid >> 7;
  const int d = c0 + cc;
  if (d < D) {
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const int rl = half * 64 + g * 32;   // first row of this 32-row group within the tile
      if (r0 + rl >= rows) break;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = tile[(rl + i) * kBothPitch + cc];
      uint4* o = reinterpret_cast<uint4*>(dstT + static_cast<long long>(d) * r_cap + r0 + rl);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        o[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                          pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
    }
  }
}

template <bool SCALE>
cudaError_t both_impl(const void* src, int D, int K, const RoutingPtrs& rp, void* dst, void* dstT, int r_cap,
                      cudaStream_t stream) {
  auto kern = gather_both_kernel<SCALE>;
  static PerDeviceOnce setup;
  const cudaError_t se =
      setup.once([&] { return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kBothSmem); });
  if (se != cudaSuccess) return se;
  dim3 grid((D + kBothCols - 1) / kBothCols, (r_cap + kBothRows - 1) / kBothRows);
  kern<<<grid, 256, kBothSmem, stream>>>(static_cast<const __nv_bfloat16*>(src), D, K, rp.hdr, rp.perm, rp.scores,
                                         static_cast<__nv_bfloat16*>(dst), static_cast<__nv_bfloat16*>(dstT), r_cap);
  return cudaGetLastError();
}

// MXFP8 variant of the same pass, one CTA per 128-row x 128-column tile.
//  * Row pass: thread t owns row t/2 and 64 contiguous columns (two MX
//    blocks) of it, so each block's scale comes from the thread's own
//    registers; the row's four scales are one 32-bit word of its atom.  The
//    BF16 values also go to shared memory for the column pass: row pitch
//    288 bytes, the two halves of a row 144 bytes apart, so the 16-byte
//    stores of a quarter-warp (4 rows x 2 halves) hit distinct banks.
//  * Column pass: thread (pair q, group g) builds features 2q and 2q+1 for
//    rows 32g .. 32g+31 from 32-bit reads (a warp reads 128 contiguous
//    bytes of one row).
// Both quantised tiles are built in shared memory as 128 x 128-byte tiles in
// the 128-byte swizzle (16-byte chunk j of line m at chunk j ^ (m % 8)) and
// leave with two TMA stores: row bundle lines are token rows
// (dst[r][c0 ..]), column bundle lines are features (dstT[d][r0 ..]).  Rows
// past the routed rows are written as zeros; nothing reads them.
constexpr int kMxPitchB = 288, kMxHalfB = 144;
constexpr int kMxSmem = 1024 + 2 * 16384 + kBothRows * kMxPitchB + kBothRows * 4;

// e4m3 codes of 32 values scaled by 2^-e, low byte first
__device__ __forceinline__ void mx_codes32(const float (&v)[32], int e, uint32_t (&w)[8]) {
  const float inv = exp2_int(-e);
#pragma unroll
  for (int k = 0; k < 8; ++k)
    w[k] = cvt_e4m3x2(v[4 * k] * inv, v[4 * k + 1] * inv) | (cvt_e4m3x2(v[4 * k + 2] * inv, v[4 * k + 3] * inv) << 16);
}

__device__ __forceinline__ float amax32(const float (&v)[32]) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(v[i]));
  return a;
}

template <bool SCALE>
__global__ void __launch_bounds__(256, 3) gather_both_mx_kernel(const __grid_constant__ CUtensorMap tm_row,
                                                                const __grid_constant__ CUtensorMap tm_col,
                                                                const __nv_bfloat16* __restrict__ src, int D, int K,
                                                                const int* __restrict__ hdr,
                                                                const int* __restrict__ perm,
                                                                const float* __restrict__ scores,
                                                                uint8_t* __restrict__ dst_sf,
                                                                uint8_t* __restrict__ dstT_sf, int b_cap,
                                                                const int* __restrict__ row_block,
                                                                const int4* __restrict__ blocks) {
  extern __shared__ uint8_t gmx_smem_raw[];
  uint8_t* rb = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gmx_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* cb = rb + 16384;
  uint8_t* xs = cb + 16384;
  float* s_row = reinterpret_cast<float*>(xs + kBothRows * kMxPitchB);
  __shared__ int s_blk[kBothRows / 32], s_b0[kBothRows / 32];
  const int rows = hdr[2];
  const int r0 = blockIdx.y * kBothRows;
  if (r0 >= rows) return;
  const int c0 = blockIdx.x * kBothCols;
  const int tid = threadIdx.x;
  if (tid < kBothRows / 32) {
    const bool in = r0 + 32 * tid < rows;
    const int b = in ? row_block[(r0 >> 5) + tid] : 0;
    s_blk[tid] = b;
    s_b0[tid] = in ? blocks[b].y : 0;
  }
  // ---- row pass
  const int row = tid >> 1, h = tid & 1;
  const int r = r0 + row;
  uint32_t sword;   // this thread's two block scales (bytes 0, 1)
  {
    const int route = r < rows ? perm[r] : -1;
    uint4 u[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) u[j] = make_uint4(0, 0, 0, 0);
    float sc = 1.0f;
    if (route >= 0) {
      const uint4* s4 = reinterpret_cast<const uint4*>(src + static_cast<long long>(route / K) * D + c0 + 64 * h);
#pragma unroll
      for (int j = 0; j < 8; ++j) u[j] = __ldg(s4 + j);
      if (SCALE) sc = scores[route];
    } else if (SCALE) {
      sc = 0.0f;
    }
    if (SCALE && h == 0) s_row[row] = sc;
    uint8_t* xrow = xs + row * kMxPitchB + h * kMxHalfB;
#pragma unroll
    for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(xrow + j * 16) = u[j];
    sword = 0;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      float v[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 w4 = u[4 * blk + q];
        const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[8 * q + 2 * k] = bf16_lo(ww[k]);
          v[8 * q + 2 * k + 1] = bf16_hi(ww[k]);
        }
      }
      if (SCALE) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= sc;
      }
      const int e = mx_shared_exp(amax32(v));
      uint32_t w[8];
      mx_codes32(v, e, w);
      // bytes 32 (2h + blk) .. +31 of the row's line: chunks 2 (2h + blk) and +1
      const int ch = 2 * (2 * h + blk);
      *reinterpret_cast<uint4*>(rb + row * 128 + ((ch ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(rb + row * 128 + (((ch + 1) ^ (row & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
      sword |= static_cast<uint32_t>(e + 127) << (8 * blk);
    }
    sword |= __shfl_xor_sync(0xFFFFFFFFu, sword, 1) << 16;   // h = 0: blocks 2, 3 from its partner
  }
  __syncthreads();
  if (h == 0 && r < rows) {
    const int p = r - s_b0[row >> 5];
    *reinterpret_cast<uint32_t*>(dst_sf + (static_cast<long long>(s_blk[row >> 5]) * (D / 128) + (c0 >> 7)) * 512 +
                                 (p & 31) * 16 + (p >> 5) * 4) = sword;
  }
  // ---- column pass
  {
    const int q = tid & 63, g = tid >> 6;
    const int rl = 32 * g;   // first row of the group within the tile
    const uint8_t* xcol = xs + (q >> 5) * kMxHalfB + (q & 31) * 4;
    uint32_t pr[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) pr[i] = *reinterpret_cast<const uint32_t*>(xcol + (rl + i) * kMxPitchB);
#pragma unroll
    for (int f = 0; f < 2; ++f) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v[i] = f == 0 ? bf16_lo(pr[i]) : bf16_hi(pr[i]);
        if (SCALE) v[i] *= s_row[rl + i];
      }
      const int e = mx_shared_exp(amax32(v));
      uint32_t w[8];
      mx_codes32(v, e, w);
      const int cc = 2 * q + f;   // feature within the slab
      *reinterpret_cast<uint4*>(cb + cc * 128 + (((2 * g) ^ (cc & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(cb + cc * 128 + (((2 * g + 1) ^ (cc & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
      if (r0 + rl < rows) {
        const int d = c0 + cc;
        const int rg = (r0 + rl) >> 5;
        dstT_sf[(static_cast<long long>(d >> 7) * b_cap + s_blk[g]) * 512 + sf_atom_byte(d & 127, rg - (s_b0[g] >> 5))] =
            static_cast<uint8_t>(e + 127);
      }
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0) {
    tma_store_2d(&tm_row, rb, c0, r0);
    tma_store_2d(&tm_col, cb, r0, c0);
    bulk_commit();
    bulk_wait_read<0>();   // the staging must outlive the stores' reads
  }
}

template <bool SCALE>
cudaError_t both_mx_impl(const CUtensorMap* tm_row, const CUtensorMap* tm_col, const void* src, int D, int K,
                         const RoutingPtrs& rp, uint8_t* dst_sf, uint8_t* dstT_sf, int r_cap, int b_cap,
                         cudaStream_t stream) {
  auto kern = gather_both_mx_kernel<SCALE>;
  static PerDeviceOnce setup;
  const cudaError_t se =
      setup.once([&] { return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMxSmem); });
  if (se != cudaSuccess) return se;
  dim3 grid(D / kBothCols, r_cap / kBothRows);
  kern<<<grid, 256, kMxSmem, stream>>>(*tm_row, *tm_col, static_cast<const __nv_bfloat16*>(src), D, K, rp.hdr,
                                       rp.perm, rp.scores, dst_sf, dstT_sf, b_cap, rp.row_block, rp.blocks);
  return cudaGetLastError();
}

template <bool MX, bool SCALE>
cudaError_t rows_impl(const void* src, int D, int K, const RoutingPtrs& rp, void* dst, uint8_t* dst_sf, int r_cap,
                      int num_sms, cudaStream_t stream) {
  const int warps_needed = r_cap;
  int blocks = (warps_needed + 7) / 8;
  blocks = min(blocks, num_sms * 8);
  gather_rows_kernel<MX, SCALE><<<blocks, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(src), D, K, rp.hdr,
                                                            rp.perm, rp.scores, dst, dst_sf, rp.row_block,
                                                            rp.blocks);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather_rows(bool mx, bool use_scores, const void* src, int D, int K, const RoutingPtrs& rp,
                               void* dst, uint8_t* dst_sf, int r_cap, int num_sms, cudaStream_t stream) {
  if (mx) {
    return use_scores ? rows_impl<true, true>(src, D, K, rp, dst, dst_sf, r_cap, num_sms, stream)
                      : rows_impl<true, false>(src, D, K, rp, dst, dst_sf, r_cap, num_sms, stream);
  }
  return use_scores ? rows_impl<false, true>(src, D, K, rp, dst, dst_sf, r_cap, num_sms, stream)
                    : rows_impl<false, false>(src, D, K, rp, dst, dst_sf, r_cap, num_sms, stream);
}

cudaError_t launch_gather_both(bool mx, bool use_scores, const void* src, int D, int K, const RoutingPtrs& rp,
                               void* dst, uint8_t* dst_sf, void* dstT, uint8_t* dstT_sf, int r_cap, int b_cap,
                               int num_sms, cudaStream_t stream, const CUtensorMap* tm_row,
                               const CUtensorMap* tm_col) {
  if (mx) {
    if (!tm_row || !tm_col || D % kBothCols != 0 || r_cap % kBothRows != 0) return cudaErrorInvalidValue;
    return use_scores ? both_mx_impl<true>(tm_row, tm_col, src, D, K, rp, dst_sf, dstT_sf, r_cap, b_cap, stream)
                      : both_mx_impl<false>(tm_row, tm_col, src, D, K, rp, dst_sf, dstT_sf, r_cap, b_cap, stream);
  }
  return use_scores ? both_impl<true>(src, D, K, rp, dst, dstT, r_cap, stream)
                    : both_impl<false>(src, D, K, rp, dst, dstT, r_cap, stream);
}

}  // namespace moe
