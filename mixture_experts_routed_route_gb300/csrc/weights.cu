// Weight preparation, run once outside any timed region.
//
// "Meta Dist-MoE: Open-Source Fused MoE Kernels for Blackwell", "Supported
// modes": prepare_block_scaled_weight quantises expert weights once, with
// 32x32 blocks for MXFP8 training-compatible values.  Dist-MoE explainer
// section 02, "Quantization Axes for Forward and Backward": with 32x32
// blocks the forward and the input-gradient GEMMs use the same quantised
// values with distinct scale orientations.  Here the one scale of each tile
// is written for both orientations and the codes once more transposed
// ([E,K,N]), so the input-gradient GEMM also reads a K-major operand.  The
// scales are written in the GEMMs' 512-byte atom layout (kernels.cuh:
// sf_atom_byte): atom (r/128, k/128) of the [E*N, K] orientation and atom
// (k/128, r/128) of the [E*K, N] one each hold 128 rows x 4 blocks of 32, so
// a GEMM stage copies one atom per operand tile in bulk.
#include "kernels.cuh"

namespace moe {

namespace {

// One CTA per (expert, 32-row block, 256-column slab); warp w owns the
// 32x32 tile at columns [32w, 32w+32) of the slab.
__global__ void __launch_bounds__(256) prep_mx_kernel(const __nv_bfloat16* __restrict__ w, int N, int K,
                                                      uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                      uint8_t* __restrict__ qT, uint8_t* __restrict__ sfT) {
  __shared__ float tile[32][257];
  __shared__ __align__(16) uint8_t qt[32][256 + 16];
  const int slabs = (K + 255) / 256;
  const int e = blockIdx.y;
  const int nb = blockIdx.x / slabs;
  const int k0 = (blockIdx.x % slabs) * 256;
  const int n0 = nb * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const __nv_bfloat16* src = w + (static_cast<long long>(e) * N + n0) * K;
  for (int i = tid; i < 32 * 32; i += 256) {
    const int row = i >> 5, chunk = i & 31;
    const int c = k0 + chunk * 8;
    if (c < K) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(src + static_cast<long long>(row) * K + c));
      tile[row][chunk * 8 + 0] = bf16_lo(u.x);
      tile[row][chunk * 8 + 1] = bf16_hi(u.x);
      tile[row][chunk * 8 + 2] = bf16_lo(u.y);
      tile[row][chunk * 8 + 3] = bf16_hi(u.y);
      tile[row][chunk * 8 + 4] = bf16_lo(u.z);
      tile[row][chunk * 8 + 5] = bf16_hi(u.z);
      tile[row][chunk * 8 + 6] = bf16_lo(u.w);
      tile[row][chunk * 8 + 7] = bf16_hi(u.w);
    }
  }
  __syncthreads();
  const int kc = k0 + warp * 32;  // first column of this warp's tile
  if (kc < K) {
    const int col = warp * 32 + lane;
    float amax = 0.0f;
#pragma unroll
    for (int r = 0; r < 32; ++r) amax = fmaxf(amax, fabsf(tile[r][col]));
    amax = warp_max_nonneg(amax);
    const int ex = mx_shared_exp(amax);
    const float inv = exp2_int(-ex);
    const uint8_t sbyte = static_cast<uint8_t>(ex + 127);
#pragma unroll
    for (int r = 0; r < 32; r += 2) {
      const uint32_t two = cvt_e4m3x2(tile[r][col] * inv, tile[r + 1][col] * inv);
      qt[r][col] = static_cast<uint8_t>(two & 0xFF);
      qt[r + 1][col] = static_cast<uint8_t>(two >> 8);
    }
    // the one scale in both orientations, as 512-byte atoms: row n of the
    // tile (K-block kc/32) in [E*N/128][K/128], and row k of the transposed
    // tile (N-block nb) in [E*K/128][N/128]
    const long long nrow = static_cast<long long>(e) * N + n0 + lane;
    const int kb = kc / 32;
    sf[((nrow >> 7) * (K / 128) + (kb >> 2)) * 512 + sf_atom_byte(static_cast<int>(nrow & 127), kb & 3)] = sbyte;
    if (sfT) {
      const long long krow = static_cast<long long>(e) * K + kc + lane;
      sfT[((krow >> 7) * (N / 128) + (nb >> 2)) * 512 + sf_atom_byte(static_cast<int>(krow & 127), nb & 3)] = sbyte;
    }
  }
  __syncthreads();
  // codes, row-major [E,N,K]
  for (int i = tid; i < 32 * 16; i += 256) {
    const int row = i >> 4, chunk = i & 15;
    const int c = k0 + chunk * 16;
    if (c < K)
      *reinterpret_cast<uint4*>(q + (static_cast<long long>(e) * N + n0 + row) * K + c) =
          *reinterpret_cast<const uint4*>(&qt[row][chunk * 16]);
  }
  // codes, transposed [E,K,N]: thread per column, 32 contiguous bytes
  if (qT) {
    const int c = k0 + tid;
    if (c < K) {
      uint32_t wv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        wv[j] = static_cast<uint32_t>(qt[4 * j][tid]) | (static_cast<uint32_t>(qt[4 * j + 1][tid]) << 8) |
                (static_cast<uint32_t>(qt[4 * j + 2][tid]) << 16) | (static_cast<uint32_t>(qt[4 * j + 3][tid]) << 24);
      uint4* o = reinterpret_cast<uint4*>(qT + (static_cast<long long>(e) * K + c) * N + n0);
      o[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      o[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
    }
  }
}

// 1x32 blocks (inference weights, "Meta Dist-MoE: Open-Source Fused MoE
// Kernels for Blackwell", "Supported modes"): thread b quantises block b of
// the flattened [rows, K/32] grid, 32 consecutive values of one row along K,
// with its own scale (same OCP rule), into the same codes / atom layout the
// 32x32 preparation writes.
__global__ void __launch_bounds__(256) prep_mx_row32_kernel(const __nv_bfloat16* __restrict__ w, long long rows,
                                                            int K, uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  const int kbs = K / 32;
  const long long nb = rows * kbs;
  for (long long b = blockIdx.x * 256LL + threadIdx.x; b < nb; b += static_cast<long long>(gridDim.x) * 256) {
    const long long row = b / kbs;
    const int kb = static_cast<int>(b - row * kbs);
    const uint4* src = reinterpret_cast<const uint4*>(w + row * K + kb * 32);
    float v[32];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 u = __ldg(src + j);
      v[8 * j + 0] = bf16_lo(u.x);
      v[8 * j + 1] = bf16_hi(u.x);
      v[8 * j + 2] = bf16_lo(u.y);
      v[8 * j + 3] = bf16_hi(u.y);
      v[8 * j + 4] = bf16_lo(u.z);
      v[8 * j + 5] = bf16_hi(u.z);
      v[8 * j + 6] = bf16_lo(u.w);
      v[8 * j + 7] = bf16_hi(u.w);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int ex = mx_shared_exp(amax);
    const float inv = exp2_int(-ex);
    uint32_t c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      c[i] = cvt_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv) | (cvt_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv) << 16);
    uint4* dst = reinterpret_cast<uint4*>(q + row * K + kb * 32);
    dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
    dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
    sf[((row >> 7) * (K / 128) + (kb >> 2)) * 512 + sf_atom_byte(static_cast<int>(row & 127), kb & 3)] =
        static_cast<uint8_t>(ex + 127);
  }
}

// BF16 [E,N,K] -> [E,K,N] through 32x32 shared-memory tiles.
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const __nv_bfloat16* __restrict__ w, int N, int K,
                                                             __nv_bfloat16* __restrict__ wT) {
  __shared__ __nv_bfloat16 t[32][33];
  const int e = blockIdx.z;
  const int n0 = blockIdx.y * 32, k0 = blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  const __nv_bfloat16* src = w + static_cast<long long>(e) * N * K;
  __nv_bfloat16* dst = wT + static_cast<long long>(e) * N * K;
  for (int r = ty; r < 32; r += 8) t[r][tx] = src[static_cast<long long>(n0 + r) * K + k0 + tx];
  __syncthreads();
  for (int r = ty; r < 32; r += 8) dst[static_cast<long long>(k0 + r) * N + n0 + tx] = t[tx][r];
}

}  // namespace

cudaError_t launch_prep_mx_weight(const void* w, int E, int N, int K, uint8_t* q, uint8_t* sf, uint8_t* qT,
                                  uint8_t* sfT, cudaStream_t stream) {
  const int slabs = (K + 255) / 256;
  dim3 grid((N / 32) * slabs, E);
  prep_mx_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(w), N, K, q, sf, qT, sfT);
  return cudaGetLastError();
}

cudaError_t launch_prep_mx_weight_row32(const void* w, int E, int N, int K, uint8_t* q, uint8_t* sf,
                                        cudaStream_t stream) {
  const long long rows = static_cast<long long>(E) * N;
  const long long blocks = (rows * (K / 32) + 255) / 256;
  const int grid = static_cast<int>(blocks < 65535 * 16 ? blocks : 65535 * 16);
  prep_mx_row32_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(w), rows, K, q, sf);
  return cudaGetLastError();
}

cudaError_t launch_transpose_bf16(const void* w, int E, int N, int K, void* wT, cudaStream_t stream) {
  dim3 grid(K / 32, N / 32, E);
  transpose_bf16_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(w), N, K,
                                                  static_cast<__nv_bfloat16*>(wT));
  return cudaGetLastError();
}

}  // namespace moe
