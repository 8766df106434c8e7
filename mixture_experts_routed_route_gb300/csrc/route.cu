// F0 routing: per-expert histogram of the active routes, exclusive prefix
// sums (plain and padded to 32 rows), a stable expert-major permutation and
// its inverse, and the list of <=128-row blocks the grouped GEMMs walk.
//
// "Mixture of Experts: How Routing Becomes GPU Computation", section 2
// "Packing": rows are sorted by expert with a stable order, an exclusive
// prefix sum of the counts gives each expert's row interval, and the inverse
// permutation is kept for the combine.  "Scheduling": the row-tile schedule
// is built on the GPU here (no host copy of the counts), so the layer stays
// capturable in a CUDA graph.  Dist-MoE explainer section 01: pad rows
// (each expert padded to its row multiple) gather zeros and scatter nowhere;
// ID -1 is an inactive route.
//
// Row-block pairs: the grouped GEMMs of dense enough routings take two
// consecutive blocks of one expert (up to 256 rows) as one B operand, so
// every tensor-core instruction is 256 wide.  Pair p of the routing is
// described in the fourth word of blocks[p]: (first block << 1) | (1 if the
// pair has a second block); the header's word 4 counts the pairs.  Each
// expert's blocks pair up in order: blocks 0+1, 2+3, ..., the last alone
// when the expert has an odd number.
//
// One CTA of 32 warps.  Warp w owns the contiguous route segment
// [w*seg, (w+1)*seg); within a warp, routes are taken 32 at a time in
// order, and lanes holding the same expert are grouped (one ballot per bit
// of the expert id), so each route's rank within its expert is (earlier
// warps' count) + (earlier batches of this warp) + (lower lanes of its
// group): exactly the stable order by flat index t*K+k.
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
// Routes per lane held in registers for both passes (read once, with all
// loads in flight together): up to kWarps * 32 * kHold = 16384 routes.
constexpr int kHold = 16;

// Lanes of the warp whose expert equals this lane's (e = -1: inactive).
// One ballot per bit of the id plus one for activity, so the cost does not
// grow with the number of distinct experts among the 32 routes, as
// match.any's does (with 64..384 experts nearly every lane differs).
__device__ __forceinline__ unsigned same_expert_lanes(int e, int nbits) {
  const bool act = e >= 0;
  const unsigned ba = __ballot_sync(0xFFFFFFFFu, act);
  unsigned m = act ? ba : ~ba;
  for (int b = 0; b < nbits; ++b) {
    const bool bit = (e >> b) & 1;
    const unsigned bb = __ballot_sync(0xFFFFFFFFu, bit);
    m &= bit ? bb : ~bb;
  }
  return m;
}

// Exclusive block-wide scan of three ints per thread (one thread per slot).
__device__ void block_scan3(int a, int b, int c, int& ea, int& eb, int& ec, int& ta, int& tb, int& tc,
                            int* ws /* [3*32] */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b, ic = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int na = __shfl_up_sync(0xFFFFFFFFu, ia, o);
    const int nb = __shfl_up_sync(0xFFFFFFFFu, ib, o);
    const int nc = __shfl_up_sync(0xFFFFFFFFu, ic, o);
    if (lane >= o) {
      ia += na;
      ib += nb;
      ic += nc;
    }
  }
  if (lane == 31) {
    ws[warp] = ia;
    ws[32 + warp] = ib;
    ws[64 + warp] = ic;
  }
  __syncthreads();
  if (warp == 0) {
    int wa = ws[lane], wb = ws[32 + lane], wc = ws[64 + lane];
    int xa = wa, xb = wb, xc = wc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int na = __shfl_up_sync(0xFFFFFFFFu, xa, o);
      const int nb = __shfl_up_sync(0xFFFFFFFFu, xb, o);
      const int nc = __shfl_up_sync(0xFFFFFFFFu, xc, o);
      if (lane >= o) {
        xa += na;
        xb += nb;
        xc += nc;
      }
    }
    __syncwarp();
    ws[lane] = xa - wa;       // exclusive prefix of warp totals
    ws[32 + lane] = xb - wb;
    ws[64 + lane] = xc - wc;
    if (lane == 31) {
      ws[96] = xa;
      ws[97] = xb;
      ws[98] = xc;
    }
  }
  __syncthreads();
  ea = ia - a + ws[warp];
  eb = ib - b + ws[32 + warp];
  ec = ic - c + ws[64 + warp];
  ta = ws[96];
  tb = ws[97];
  tc = ws[98];
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
    route_kernel(const int32_t* __restrict__ ids, const float* __restrict__ scores, int T, int K, int E,
                 int r_cap, int debug, RoutingPtrs rp, uint32_t* __restrict__ err) {
  extern __shared__ int sm[];
  int* hist = sm;                 // [kWarps][E]: counts, then running row bases
  int* s_cnt = hist + kWarps * E; // [E]
  int* s_poff = s_cnt + E;        // [E + 1]
  __shared__ int ws[128];
  __shared__ unsigned s_err;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int TK = T * K;
  const int seg = (TK + kWarps - 1) / kWarps;
  const int beg = min(warp * seg, TK), end = min(beg + seg, TK);
  if (tid == 0) s_err = 0;
  for (int i = tid; i < kWarps * E; i += kThreads) hist[i] = 0;
  __syncthreads();

  // ---- pass 1: per-warp histograms (and validation of the IDs)
  int* myh = hist + warp * E;
  unsigned my_err = 0;
  const bool held = seg <= 32 * kHold;
  int idr[kHold];
  if (held) {
#pragma unroll
    for (int j = 0; j < kHold; ++j) {
      const int i = beg + 32 * j + lane;
      idr[j] = i < end ? ids[i] : -1;
    }
  }
  // the saved copy of the scores, while the ID loads are in flight: 16-byte
  // vectors, every load issued at once (pass 3 zeroes the inactive routes'
  // entries after the barriers below), so the scatter issues no loads
  if ((reinterpret_cast<uintptr_t>(scores) & 15) == 0) {   // the caller's scores need only 4-byte alignment
    const int n4 = TK / 4;
    const float4* s4 = reinterpret_cast<const float4*>(scores);
    float4* d4 = reinterpret_cast<float4*>(rp.scores);
    for (int q = tid; q < n4; q += kThreads) d4[q] = s4[q];
    if (tid < TK - 4 * n4) rp.scores[4 * n4 + tid] = scores[4 * n4 + tid];
  } else {
    for (int i = tid; i < TK; i += kThreads) rp.scores[i] = scores[i];
  }
  // expert of route i with id `id` (-1: inactive), flagging bad IDs
  auto classify = [&](int i, int id) {
    if (id >= 0 && id < E) return id;
    if (id != -1) my_err |= kErrBadId;
    else if (debug && scores[i] != 0.0f) my_err |= kErrInactiveScore;
    return -1;
  };
  // counts need no order: one shared-memory atomic per active route
  auto count = [&](int e) {
    if (e >= 0) atomicAdd(&myh[e], 1);
  };
  if (held) {
#pragma unroll
    for (int j = 0; j < kHold; ++j) {
      if (beg + 32 * j < end) {
        const int i = beg + 32 * j + lane;
        count(i < end ? classify(i, idr[j]) : -1);
      }
    }
  } else {
    for (int base = beg; base < end; base += 32) {
      const int i = base + lane;
      count(i < end ? classify(i, ids[i]) : -1);
    }
  }
  if (my_err) atomicOr(&s_err, my_err);
  __syncthreads();

  // ---- pass 2: counts, exclusive prefixes (plain, padded, block counts)
  int c = 0;
  if (tid < E) {
    for (int w = 0; w < kWarps; ++w) c += hist[w * E + tid];
    s_cnt[tid] = c;
  }
  const int pc = (c + kPad - 1) / kPad * kPad;
  const int nb = (pc + kBlockRows - 1) / kBlockRows;
  int eo, ep, eb, to, tp, tb, epr, tpr, d0, d1, d2, d3;
  block_scan3(tid < E ? c : 0, tid < E ? pc : 0, tid < E ? nb : 0, eo, ep, eb, to, tp, tb, ws);
  const int np = (nb + 1) / 2;
  block_scan3(tid < E ? np : 0, 0, 0, epr, d0, d1, tpr, d2, d3, ws);
  if (tid < E) {
    rp.counts[tid] = c;
    rp.offsets[tid] = eo;
    rp.poffsets[tid] = ep;
    s_poff[tid] = ep;
    // running row base of each warp for this expert
    int run = ep;
    for (int w = 0; w < kWarps; ++w) {
      const int h = hist[w * E + tid];
      hist[w * E + tid] = run;
      run += h;
    }
    // row blocks of this expert, and the block of each of its 32-row groups
    rp.bstart[tid] = eb;
    for (int b = 0; b < nb; ++b) {
      const int rows_b = min(kBlockRows, pc - b * kBlockRows);
      rp.blocks[eb + b] = make_int4(tid, ep + b * kBlockRows, rows_b, 0);
      for (int g = 0; g < rows_b / kPad; ++g) rp.row_block[(ep + b * kBlockRows) / kPad + g] = eb + b;
    }
  }
  if (tid == 0) {
    rp.offsets[E] = to;
    rp.poffsets[E] = tp;
    rp.bstart[E] = tb;
    s_poff[E] = tp;
    rp.hdr[0] = T;
    rp.hdr[1] = tb;
    rp.hdr[2] = tp;
    rp.hdr[3] = to;
    rp.hdr[4] = tpr;
  }
  __syncthreads();
  // pair descriptors, once every block entry is written
  if (tid < E) {
    for (int q = 0; q < np; ++q)
      reinterpret_cast<int*>(rp.blocks + epr + q)[3] = ((eb + 2 * q) << 1) | (2 * q + 1 < nb ? 1 : 0);
  }

  // ---- pass 3: stable scatter of each route to its row
  const int nbits = E > 1 ? 32 - __clz(E - 1) : 0;
  auto scatter = [&](int i, int id) {
    const int e = (i < end && id >= 0 && id < E) ? id : -1;
    const unsigned grp = same_expert_lanes(e, nbits);
    const unsigned lower = grp & ((1u << lane) - 1u);
    if (e >= 0) {
      const int row = myh[e] + __popc(lower);
      rp.perm[row] = i;
      rp.inv[i] = row;
    } else if (i < end) {
      rp.inv[i] = -1;
      rp.scores[i] = 0.0f;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(grp) - 1) myh[e] += __popc(grp);
    __syncwarp();
  };
  if (held) {
#pragma unroll
    for (int j = 0; j < kHold; ++j)
      if (beg + 32 * j < end) scatter(beg + 32 * j + lane, idr[j]);
  } else {
    for (int base = beg; base < end; base += 32) {
      const int i = base + lane;
      scatter(i, i < end ? ids[i] : -1);
    }
  }

  // ---- pass 4: pad rows and the unused tail of the row capacity
  for (int j = tid; j < E * kPad; j += kThreads) {
    const int e = j / kPad, k = j % kPad;
    const int row = s_poff[e] + s_cnt[e] + k;
    if (row < s_poff[e + 1]) rp.perm[row] = -1;
  }
  for (int row = s_poff[E] + tid; row < r_cap; row += kThreads) rp.perm[row] = -1;

  __syncthreads();
  if (tid == 0 && s_err) atomicOr(err, s_err);
}

}  // namespace

cudaError_t launch_route(const int32_t* ids, const float* scores, int T, int K, int E, int r_cap, int debug,
                         const RoutingPtrs& rp, uint32_t* err, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(kWarps * E + E + E + 1) * sizeof(int);
  // the opt-in covers the largest expert count a context accepts (1024), so
  // one set-up per device serves every launch
  static PerDeviceOnce setup;
  if (smem > 48 * 1024) {
    const int max_smem = (kWarps * 1024 + 1024 + 1024 + 1) * static_cast<int>(sizeof(int));
    const cudaError_t se = setup.once(
        [&] { return cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem); });
    if (se != cudaSuccess) return se;
  }
  route_kernel<<<1, kThreads, smem, stream>>>(ids, scores, T, K, E, r_cap, debug, rp, err);
  return cudaGetLastError();
}

}  // namespace moe
