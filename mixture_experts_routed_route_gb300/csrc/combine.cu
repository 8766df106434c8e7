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
#include "kernels.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16* __restrict__ h, int D, int K,
                                                      const int* __restrict__ inv, const float* __restrict__ scores,
                                                      __nv_bfloat16* __restrict__ out, int T, int accumulate,
                                                      const int* __restrict__ hdr) {
  if (hdr) T = min(T, hdr[0]);
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    for (int c = threadIdx.x * 8; c < D; c += blockDim.x * 8) {
      float acc[8];
      __nv_bfloat16* o = out + static_cast<long long>(t) * D + c;
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
      for (int k = 0; k < K; ++k) {
        const int r = inv[t * K + k];
        if (r < 0) continue;
        const float s = scores ? scores[t * K + k] : 1.0f;
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(h + static_cast<long long>(r) * D + c));
        acc[0] = fmaf(s, bf16_lo(u.x), acc[0]);
        acc[1] = fmaf(s, bf16_hi(u.x), acc[1]);
        acc[2] = fmaf(s, bf16_lo(u.y), acc[2]);
        acc[3] = fmaf(s, bf16_hi(u.y), acc[3]);
        acc[4] = fmaf(s, bf16_lo(u.z), acc[4]);
        acc[5] = fmaf(s, bf16_hi(u.z), acc[5]);
        acc[6] = fmaf(s, bf16_lo(u.w), acc[6]);
        acc[7] = fmaf(s, bf16_hi(u.w), acc[7]);
      }
      *reinterpret_cast<uint4*>(o) = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                                pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
  }
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
                           bool accumulate, int num_sms, cudaStream_t stream, const int* hdr) {
  if (T <= 0) return cudaSuccess;
  const int threads = min(256, max(32, (D / 8 + 31) / 32 * 32));
  const int blocks = min(T, num_sms * 16);
  combine_kernel<<<blocks, threads, 0, stream>>>(static_cast<const __nv_bfloat16*>(h), D, K, inv, scores,
                                                 static_cast<__nv_bfloat16*>(out), T, accumulate ? 1 : 0, hdr);
  return cudaGetLastError();
}

}  // namespace moe
