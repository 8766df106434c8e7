// F1 / B0: gather token rows into expert-major order, optionally scaled by
// the route's score, as BF16 or as MXFP8 (E4M3 + one E8M0 scale per 32
// values).
//
// Dist-MoE explainer section 02, "Quantization Axes for Forward and
// Backward": FPROP/DGRAD operands are scaled along the feature axis (row
// bundles, launch_gather_rows); WGRAD contracts over token rows and needs a
// separately quantised column-oriented bundle (stored transposed [D, r_cap]
// so the GEMM reads it K-major); launch_gather_both writes both bundles of
// the same rows in one pass when training.  MXFP8 training
// quantises after the gather ("MXFP8 training publishes BF16 source rows and
// quantizes after peer gather"); row quantisation depends only on the row,
// so quantising after the gather is exact.  Pad rows (route -1) are zero.
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
    for (int base = 0; base < D; base += 256) {
      const int c = base + lane * 8;
      const bool act = c < D;
      uint4 u = make_uint4(0, 0, 0, 0);
      if (act && srow) u = __ldg(reinterpret_cast<const uint4*>(srow + c));
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

// Both bundles in one pass (training).  One CTA per (128-row tile,
// 128-column slab): the gathered rows go through shared memory once, then
//  * row bundle: warp w writes rows 16w .. 16w+15, lane l columns 4l .. 4l+3
//    (8 lanes per MX block; 128 contiguous bytes per row and warp);
//  * column bundle: thread (c, half) writes feature c0+c for rows
//    64*half .. +63, i.e. 64 contiguous bytes (two MX blocks) per thread, so
//    two threads fill each 128-byte line of dstT[feature][rows] at once.
constexpr int kBothRows = 128, kBothCols = 128, kBothPitch = kBothCols + 4;
constexpr int kBothSmem = kBothRows * kBothPitch * 4;

template <bool MX, bool SCALE>
__global__ void __launch_bounds__(256) gather_both_kernel(const __nv_bfloat16* __restrict__ src, int D, int K,
                                                          const int* __restrict__ hdr, const int* __restrict__ perm,
                                                          const float* __restrict__ scores, void* __restrict__ dst,
                                                          uint8_t* __restrict__ dst_sf, void* __restrict__ dstT,
                                                          uint8_t* __restrict__ dstT_sf, int r_cap, int b_cap,
                                                          const int* __restrict__ row_block,
                                                          const int4* __restrict__ blocks) {
  extern __shared__ float4 smem_f4[];
  float* tile = reinterpret_cast<float*>(smem_f4);  // [128][kBothPitch]
  const int rows = hdr[2];
  const int r0 = blockIdx.y * kBothRows;
  if (r0 >= rows) return;
  const int c0 = blockIdx.x * kBothCols;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // ---- load 128 gathered rows x 128 columns (16 chunks of 8 values per row)
  for (int i = tid; i < kBothRows * 16; i += 256) {
    const int row = i >> 4, chunk = i & 15;
    const int c = c0 + chunk * 8;
    float v[8];
    const int route = (r0 + row < r_cap) ? perm[r0 + row] : -1;
    if (route >= 0 && c < D) {
      unpack8(__ldg(reinterpret_cast<const uint4*>(src + static_cast<long long>(route / K) * D + c)), v);
      if (SCALE) {
        const float s = scores[route];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = s * v[j];
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.0f;
    }
    float4* t4 = reinterpret_cast<float4*>(tile + row * kBothPitch + chunk * 8);
    t4[0] = make_float4(v[0], v[1], v[2], v[3]);
    t4[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
  __syncthreads();
  // ---- row bundle
  const int c = c0 + lane * 4;
  for (int rr = 0; rr < 16; ++rr) {
    const int row = warp * 16 + rr;
    const int r = r0 + row;
    const float4 x4 = *reinterpret_cast<const float4*>(tile + row * kBothPitch + lane * 4);
    if (!MX) {
      if (c < D && r < rows)
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(dst) + static_cast<long long>(r) * D + c) =
            make_uint2(pack_bf16x2(x4.x, x4.y), pack_bf16x2(x4.z, x4.w));
    } else {
      float amax = fmaxf(fmaxf(fabsf(x4.x), fabsf(x4.y)), fmaxf(fabsf(x4.z), fabsf(x4.w)));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
      const int e = mx_shared_exp(amax);
      const float inv = exp2_int(-e);
      const uint32_t q = cvt_e4m3x2(x4.x * inv, x4.y * inv) | (cvt_e4m3x2(x4.z * inv, x4.w * inv) << 16);
      if (c < D && r < rows) {
        *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(dst) + static_cast<long long>(r) * D + c) = q;
        if ((lane & 7) == 0) {
          const int b = row_block[r >> 5];
          const int kb = c >> 5;
          dst_sf[(static_cast<long long>(b) * (D / 128) + (kb >> 2)) * 512 + sf_atom_byte(r - blocks[b].y, kb & 3)] =
              static_cast<uint8_t>(e + 127);
        }
      }
    }
  }
  // ---- column bundle
  const int cc = tid & 127, half = tid >> 7;
  const int d = c0 + cc;
  if (d < D) {
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const int rl = half * 64 + g * 32;   // first row of this 32-row group within the tile
      const int rg = (r0 + rl) >> 5;
      if (r0 + rl >= rows) break;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = tile[(rl + i) * kBothPitch + cc];
      if (!MX) {
        uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dstT) + static_cast<long long>(d) * r_cap + r0 + rl);
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
        uint4* o = reinterpret_cast<uint4*>(static_cast<uint8_t*>(dstT) + static_cast<long long>(d) * r_cap + r0 + rl);
        o[0] = make_uint4(w[0], w[1], w[2], w[3]);
        o[1] = make_uint4(w[4], w[5], w[6], w[7]);
        const int b = row_block[rg];
        dstT_sf[(static_cast<long long>(d >> 7) * b_cap + b) * 512 + sf_atom_byte(d & 127, rg - (blocks[b].y >> 5))] =
            static_cast<uint8_t>(e + 127);
      }
    }
  }
}

template <bool MX, bool SCALE>
cudaError_t both_impl(const void* src, int D, int K, const RoutingPtrs& rp, void* dst, uint8_t* dst_sf, void* dstT,
                      uint8_t* dstT_sf, int r_cap, int b_cap, int /*num_sms*/, cudaStream_t stream) {
  auto kern = gather_both_kernel<MX, SCALE>;
  static bool configured = false;
  if (!configured) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kBothSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid((D + kBothCols - 1) / kBothCols, (r_cap + kBothRows - 1) / kBothRows);
  kern<<<grid, 256, kBothSmem, stream>>>(static_cast<const __nv_bfloat16*>(src), D, K, rp.hdr, rp.perm, rp.scores,
                                         dst, dst_sf, dstT, dstT_sf, r_cap, b_cap, rp.row_block, rp.blocks);
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
                               int num_sms, cudaStream_t stream) {
  if (mx) {
    return use_scores ? both_impl<true, true>(src, D, K, rp, dst, dst_sf, dstT, dstT_sf, r_cap, b_cap, num_sms, stream)
                      : both_impl<true, false>(src, D, K, rp, dst, dst_sf, dstT, dstT_sf, r_cap, b_cap, num_sms, stream);
  }
  return use_scores ? both_impl<false, true>(src, D, K, rp, dst, dst_sf, dstT, dstT_sf, r_cap, b_cap, num_sms, stream)
                    : both_impl<false, false>(src, D, K, rp, dst, dst_sf, dstT, dstT_sf, r_cap, b_cap, num_sms, stream);
}

}  // namespace moe
