// F4 combine and B6 input-gradient reduction: one output row per token,
// summing the token's K route rows in a fixed order in FP32 and rounding
// once to BF16.  No atomics, so the result is bitwise reproducible.
//
// Dist-MoE explainer section 01, "Expert Gather, Scatter, and Combine": the
// owner applies its scores and sums the K routes in FP32; an all-inactive
// row returns exact zero.  "Mixture of Experts: How Routing Becomes GPU
// Computation", section 2, "SwiGLU forward": out[t] accumulates
// p(t,e) * expert output in FP32 and is cast back; "SwiGLU backward": the
// input-gradient contributions are added at their original token positions.
//
// Post-expert RMSNorm ("Meta Dist-MoE: Open-Source Fused MoE Kernels for
// Blackwell", "Supported modes", names it without defining it; reading: the
// layer's output row x, the BF16 result above, is normalised over D with a
// per-feature gamma): the combine writes x (to the saved pre-norm rows when
// training, else in place) while summing its squares, then rewrites the row
// as bf16(gamma x r), r = 1/sqrt(mean x^2 + eps).  The backward kernels give
// dx = bf16(r g - x r^3 c), g = gamma dy, c = mean(g x), and dgamma =
// sum_t dy x r through 64-token partial sums added in slab order.
#include "kernels.cuh"

namespace moe {

namespace {

// CTA-wide sum of one float per thread in a fixed order: xor trees within
// the warps, then the warp sums in warp order; every thread gets the total.
// blockDim.x is a multiple of 32.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();   // the previous call's readers are done with red
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.0f;
  for (int w = 0; w < nw; ++w) t += red[w];
  return t;
}

__device__ __forceinline__ void unpack8f(const uint4 u, float (&v)[8]) {
  v[0] = bf16_lo(u.x);
  v[1] = bf16_hi(u.x);
  v[2] = bf16_lo(u.y);
  v[3] = bf16_hi(u.y);
  v[4] = bf16_lo(u.z);
  v[5] = bf16_hi(u.z);
  v[6] = bf16_lo(u.w);
  v[7] = bf16_hi(u.w);
}

template <bool NORM>
__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16* __restrict__ h, int D, int K,
                                                      const int* __restrict__ inv, const float* __restrict__ scores,
                                                      __nv_bfloat16* __restrict__ out, int T, int accumulate,
                                                      const int* __restrict__ hdr,
                                                      const __nv_bfloat16* __restrict__ gamma, float eps,
                                                      __nv_bfloat16* __restrict__ xsave) {
  __shared__ float red[32];
  if (hdr) T = min(T, hdr[0]);
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    __nv_bfloat16* orow = out + static_cast<long long>(t) * D;
    // NORM: x goes to the saved pre-norm row, or in place (each thread
    // re-reads only its own chunks)
    __nv_bfloat16* xrow = (NORM && xsave) ? xsave + static_cast<long long>(t) * D : orow;
    float ss = 0.0f;
    for (int c = threadIdx.x * 8; c < D; c += blockDim.x * 8) {
      float acc[8];
      __nv_bfloat16* o = orow + c;
      if (accumulate) {
        const uint4 u = *reinterpret_cast<const uint4*>(o);
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
      // up to 8 routes at a time: every row load in flight before the FMAs,
      // which still run in ascending k (inactive routes skipped)
      for (int k0 = 0; k0 < K; k0 += 8) {
        int r[8];
        uint4 u[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          r[j] = k0 + j < K ? inv[t * K + k0 + j] : -1;
          u[j] = make_uint4(0, 0, 0, 0);
          if (r[j] >= 0) u[j] = __ldg(reinterpret_cast<const uint4*>(h + static_cast<long long>(r[j]) * D + c));
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (r[j] < 0) continue;
          const float s = scores ? scores[t * K + k0 + j] : 1.0f;
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
      const uint4 xv = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                  pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
      *reinterpret_cast<uint4*>(xrow + c) = xv;
      if (NORM) {
        float xf[8];
        unpack8f(xv, xf);
#pragma unroll
        for (int j = 0; j < 8; ++j) ss = fmaf(xf[j], xf[j], ss);
      }
    }
    if (NORM) {
      const float r = 1.0f / sqrtf(block_sum(ss, red) / static_cast<float>(D) + eps);
      for (int c = threadIdx.x * 8; c < D; c += blockDim.x * 8) {
        float xf[8], gf[8];
        unpack8f(*reinterpret_cast<const uint4*>(xrow + c), xf);
        unpack8f(__ldg(reinterpret_cast<const uint4*>(gamma + c)), gf);
#pragma unroll
        for (int j = 0; j < 8; ++j) xf[j] = gf[j] * (xf[j] * r);
        *reinterpret_cast<uint4*>(orow + c) = make_uint4(pack_bf16x2(xf[0], xf[1]), pack_bf16x2(xf[2], xf[3]),
                                                         pack_bf16x2(xf[4], xf[5]), pack_bf16x2(xf[6], xf[7]));
      }
    }
  }
}

// Post-norm backward, one CTA per token row: r from the saved x, then
// dx = bf16(r g - x r^3 c) with g = gamma dy, c = mean(g x); r goes to
// rstd[t] for the dgamma sums.
__global__ void __launch_bounds__(256) post_norm_bwd_kernel(const __nv_bfloat16* __restrict__ x,
                                                            const __nv_bfloat16* __restrict__ gamma,
                                                            const __nv_bfloat16* __restrict__ dy, int D, float eps,
                                                            __nv_bfloat16* __restrict__ dx, float* __restrict__ rstd,
                                                            int T, const int* __restrict__ hdr) {
  __shared__ float red[32];
  T = min(T, hdr[0]);
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const long long base = static_cast<long long>(t) * D;
    float sx = 0.0f, sgx = 0.0f;
    for (int c = threadIdx.x * 8; c < D; c += blockDim.x * 8) {
      float xf[8], gf[8], df[8];
      unpack8f(__ldg(reinterpret_cast<const uint4*>(x + base + c)), xf);
      unpack8f(__ldg(reinterpret_cast<const uint4*>(gamma + c)), gf);
      unpack8f(__ldg(reinterpret_cast<const uint4*>(dy + base + c)), df);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        sx = fmaf(xf[j], xf[j], sx);
        sgx = fmaf(gf[j] * df[j], xf[j], sgx);
      }
    }
    const float tx = block_sum(sx, red);
    const float tg = block_sum(sgx, red);
    const float r = 1.0f / sqrtf(tx / static_cast<float>(D) + eps);
    const float r3c = r * r * r * (tg / static_cast<float>(D));
    if (threadIdx.x == 0) rstd[t] = r;
    for (int c = threadIdx.x * 8; c < D; c += blockDim.x * 8) {
      float xf[8], gf[8], df[8];
      unpack8f(__ldg(reinterpret_cast<const uint4*>(x + base + c)), xf);
      unpack8f(__ldg(reinterpret_cast<const uint4*>(gamma + c)), gf);
      unpack8f(__ldg(reinterpret_cast<const uint4*>(dy + base + c)), df);
#pragma unroll
      for (int j = 0; j < 8; ++j) xf[j] = r * (gf[j] * df[j]) - xf[j] * r3c;
      *reinterpret_cast<uint4*>(dx + base + c) = make_uint4(pack_bf16x2(xf[0], xf[1]), pack_bf16x2(xf[2], xf[3]),
                                                            pack_bf16x2(xf[4], xf[5]), pack_bf16x2(xf[6], xf[7]));
    }
  }
}

// partial[s][d] = sum over the tokens of slab s, ascending, of dy x r; a
// thread owns 8 columns of one slab.  Slabs past T write zeros.
__global__ void __launch_bounds__(256) dgamma_partial_kernel(const __nv_bfloat16* __restrict__ x,
                                                             const __nv_bfloat16* __restrict__ dy,
                                                             const float* __restrict__ rstd, int D, int T,
                                                             float* __restrict__ partial,
                                                             const int* __restrict__ hdr) {
  T = min(T, hdr[0]);
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (c >= D) return;
  const int t0 = blockIdx.y * kPostNormSlab, t1 = min(T, t0 + kPostNormSlab);
  float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
  for (int t = t0; t < t1; ++t) {
    const long long base = static_cast<long long>(t) * D + c;
    float xf[8], df[8];
    unpack8f(__ldg(reinterpret_cast<const uint4*>(x + base)), xf);
    unpack8f(__ldg(reinterpret_cast<const uint4*>(dy + base)), df);
    const float r = rstd[t];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = fmaf(df[j] * xf[j], r, acc[j]);
  }
  float4* o = reinterpret_cast<float4*>(partial + static_cast<long long>(blockIdx.y) * D + c);
  o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// dgamma[d] = sum of the used slabs' partials, in slab order.
__global__ void __launch_bounds__(256) dgamma_sum_kernel(const float* __restrict__ partial, int D, int T,
                                                         float* __restrict__ dgamma, const int* __restrict__ hdr) {
  T = min(T, hdr[0]);
  const int d = blockIdx.x * blockDim.x + threadIdx.x;
  if (d >= D) return;
  const int slabs = (T + kPostNormSlab - 1) / kPostNormSlab;
  float s = 0.0f;
  for (int k = 0; k < slabs; ++k) s += partial[static_cast<long long>(k) * D + d];
  dgamma[d] = s;
}

// Score gradient ("Mixture of Experts: How Routing Becomes GPU Computation",
// section 2, "SwiGLU backward": dp(t,e) = <H(t,e), dY(t)>): one warp per
// route, each lane sums its 8-value slices in order, then a fixed xor tree.
__global__ void __launch_bounds__(256) score_grad_kernel(const __nv_bfloat16* __restrict__ h3,
                                                         const __nv_bfloat16* __restrict__ dY, int D, int K,
                                                         const int* __restrict__ inv, float* __restrict__ dp, int T,
                                                         const int* __restrict__ hdr) {
  if (hdr) T = min(T, hdr[0]);
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < T * K; i += warps) {
    const int r = inv[i];
    float acc = 0.0f;
    if (r >= 0) {
      const __nv_bfloat16* a = h3 + static_cast<long long>(r) * D;
      const __nv_bfloat16* b = dY + static_cast<long long>(i / K) * D;
      for (int c = lane * 8; c < D; c += 256) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(a + c));
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(b + c));
        acc = fmaf(bf16_lo(u.x), bf16_lo(v.x), acc);
        acc = fmaf(bf16_hi(u.x), bf16_hi(v.x), acc);
        acc = fmaf(bf16_lo(u.y), bf16_lo(v.y), acc);
        acc = fmaf(bf16_hi(u.y), bf16_hi(v.y), acc);
        acc = fmaf(bf16_lo(u.z), bf16_lo(v.z), acc);
        acc = fmaf(bf16_hi(u.z), bf16_hi(v.z), acc);
        acc = fmaf(bf16_lo(u.w), bf16_lo(v.w), acc);
        acc = fmaf(bf16_hi(u.w), bf16_hi(v.w), acc);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    }
    if (lane == 0) dp[i] = acc;
  }
}

}  // namespace

cudaError_t launch_score_grad(const void* h3, const void* dY, int D, int K, const int* inv, float* dp, int T,
                              int num_sms, cudaStream_t stream, const int* hdr) {
  if (T <= 0) return cudaSuccess;
  const int blocks = max(1, min((T * K + 7) / 8, num_sms * 8));
  score_grad_kernel<<<blocks, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(h3),
                                                static_cast<const __nv_bfloat16*>(dY), D, K, inv, dp, T, hdr);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* h, int D, int K, const int* inv, const float* scores, void* out, int T,
                           bool accumulate, int num_sms, cudaStream_t stream, const int* hdr, const void* gamma,
                           float eps, void* xsave) {
  if (T <= 0) return cudaSuccess;
  // 128-thread CTAs: at T = 2048 every token's CTA is resident in one wave
  // (16 per SM), where 256-thread CTAs took two (combine at D = 7168: 0.041
  // to 0.039 ms; the bits do not change, each thread keeps its columns)
  const int threads = min(128, max(32, (D / 8 + 31) / 32 * 32));
  const int blocks = min(T, num_sms * 16);
  const auto* hp = static_cast<const __nv_bfloat16*>(h);
  auto* op = static_cast<__nv_bfloat16*>(out);
  if (gamma) {
    combine_kernel<true><<<blocks, threads, 0, stream>>>(hp, D, K, inv, scores, op, T, accumulate ? 1 : 0, hdr,
                                                         static_cast<const __nv_bfloat16*>(gamma), eps,
                                                         static_cast<__nv_bfloat16*>(xsave));
  } else {
    combine_kernel<false><<<blocks, threads, 0, stream>>>(hp, D, K, inv, scores, op, T, accumulate ? 1 : 0, hdr,
                                                          nullptr, 0.0f, nullptr);
  }
  return cudaGetLastError();
}

cudaError_t launch_post_norm_backward(const void* x, const void* gamma, const void* dy, int D, float eps, void* dx,
                                      float* rstd, float* partial, float* dgamma, int T, int num_sms,
                                      cudaStream_t stream, const int* hdr) {
  if (T <= 0) return cudaSuccess;
  const int threads = min(256, max(32, (D / 8 + 31) / 32 * 32));
  post_norm_bwd_kernel<<<min(T, num_sms * 16), threads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(gamma),
      static_cast<const __nv_bfloat16*>(dy), D, eps, static_cast<__nv_bfloat16*>(dx), rstd, T, hdr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 pg((D / 8 + 255) / 256, (T + kPostNormSlab - 1) / kPostNormSlab);
  dgamma_partial_kernel<<<pg, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x),
                                                static_cast<const __nv_bfloat16*>(dy), rstd, D, T, partial, hdr);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dgamma_sum_kernel<<<(D + 255) / 256, 256, 0, stream>>>(partial, D, T, dgamma, hdr);
  return cudaGetLastError();
}

}  // namespace moe
