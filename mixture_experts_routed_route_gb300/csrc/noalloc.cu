// Allocation-free inference forward: moe_forward_static_scratch.
//
// Some callers cannot allocate device memory when they need the layer: an
// inference engine that hands all free HBM to its KV cache at start-up, a
// plugin that is given a stream but no allocator, or a latency-critical loop
// that must not call cudaMalloc because it can synchronise the whole device.
// This entry point runs the same kernels as the inference moe_forward
// (route, gather, W13 + SwiGLU, W2, combine) but keeps every intermediate in
// one file-scope device array instead of a context's cudaMalloc'd scratch.
//
// The GEMMs get the same tensor maps, tile pairing and grids as in
// moe_forward, so the output equals an inference moe_forward's bit for bit.
//
// The array (kStaticScratchBytes) exists on every GPU that loads the library
// and stays allocated until the process exits.  Every call shares it and it
// keeps the previous call's contents; the routing kernel rewrites every
// routing array it reads and the gather rewrites every row the GEMMs read, so
// nothing in it needs clearing.  Device errors go to the caller's error word.
// Calls that may overlap on the GPU (different streams, or different host
// threads without ordering) race on the array.
#include <mutex>

#include "kernels.cuh"
#include "moe_gb300.h"

using namespace moe;

namespace {

constexpr size_t kStaticScratchBytes = 64ull << 20;  // 64 MiB, see MOE_STATIC_SCRATCH_BYTES
constexpr size_t kAl = 256;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

struct DeviceSetup {
  bool ready = false;
  uint8_t* scratch = nullptr;  // device address of g_static_scratch on this device
  int sms = 0;
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mu;

size_t al(size_t x) { return (x + kAl - 1) / kAl * kAl; }

// Host code may not use g_static_scratch as a device address (it names a
// host-side shadow); the device address comes from cudaGetSymbolAddress,
// taken once per device with that device current.
moe_status setup_device(DeviceSetup** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  DeviceSetup& s = g_setup[dev];
  if (!s.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
    s.scratch = static_cast<uint8_t*>(p);
    s.sms = sms;
    s.ready = true;
  }
  *out = &s;
  return MOE_OK;
}

bool is16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool weight_matches(const moe_weight* w, moe_precision prec, int E, int N, int K) {
  const bool prec_ok = w && (w->precision == prec || (prec == MOE_MXFP8 && w->precision == MOE_MXFP8_1X32));
  return prec_ok && w->E == E && w->N == N && w->K == K && w->data && is16(w->data) &&
         (prec != MOE_MXFP8 || (w->scale && is16(w->scale)));
}

// Offsets of the call's buffers inside the static array.
struct StaticLayout {
  size_t hdr, counts, offsets, poffsets, perm, inv, blocks, scores, bstart, row_block;
  size_t xrow, xrow_sf, h2row, h2row_sf, h3, total;
  int64_t r_cap, b_cap;
};

// At most min(E, T*K) experts receive rows, and each pads its rows to a
// multiple of 32, so T*K + 31*min(E, T*K) rows hold every routing of T
// tokens (a one-token decode step at E = 384, K = 6 needs 192 rows, not
// the 11,910 a bound with 31*E would reserve); each receiving expert adds
// at most one partial 128-row block.
StaticLayout static_layout(int T, int D, int F, int E, int K, bool mx) {
  StaticLayout L{};
  const int64_t routes = static_cast<int64_t>(T) * K;
  const int64_t busy = routes < E ? routes : E;
  const int64_t rows = routes + 31LL * busy;
  L.r_cap = (rows + 127) / 128 * 128 + 128;
  L.b_cap = rows / 128 + busy + 1;
  const size_t esz = mx ? 1 : 2;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += al(bytes);
    return at;
  };
  L.hdr = take(16 * sizeof(int));
  L.counts = take(E * sizeof(int));
  L.offsets = take((E + 1) * sizeof(int));
  L.poffsets = take((E + 1) * sizeof(int));
  L.perm = take(L.r_cap * sizeof(int));
  L.inv = take(routes * sizeof(int));
  L.blocks = take(L.b_cap * 4 * sizeof(int));
  L.scores = take(routes * sizeof(float));
  L.bstart = take((E + 1) * sizeof(int));
  L.row_block = take((L.r_cap / 32) * sizeof(int));
  L.xrow = take(L.r_cap * D * esz);
  L.xrow_sf = mx ? take(L.b_cap * (D / 128) * 512) : 0;
  L.h2row = take(L.r_cap * F * esz);
  L.h2row_sf = mx ? take(L.b_cap * (F / 128) * 512) : 0;
  L.h3 = take(L.r_cap * D * 2);
  L.total = o;
  return L;
}

}  // namespace

extern "C" moe_status moe_forward_static_scratch(const moe_config* cfg, int32_t T, const void* x,
                                                 const int32_t* topk_ids, const float* topk_scores,
                                                 const moe_weight* W13, const moe_weight* W2, void* out,
                                                 uint32_t call_flags, uint32_t* device_error_word,
                                                 cudaStream_t stream) {
  if (!cfg || T < 0) return MOE_ERR_INVALID_ARG;
  const int D = cfg->d_model, F = cfg->d_ff, E = cfg->num_experts, K = cfg->top_k;
  if (K < 1 || K > 32 || E < 1 || E > 1024 || D < 128 || F < 128) return MOE_ERR_INVALID_ARG;
  if (cfg->precision != MOE_BF16 && cfg->precision != MOE_MXFP8) return MOE_ERR_INVALID_ARG;
  if (!(cfg->swiglu_limit >= 0.0f) || cfg->swiglu_limit > 3.0e38f) return MOE_ERR_INVALID_ARG;
  if (D % 128 || F % 128) return MOE_ERR_UNSUPPORTED;
  if (cfg->flags & MOE_POST_NORM) return MOE_ERR_UNSUPPORTED;   // its gamma lives in a context
  if (call_flags & ~MOE_ACCUMULATE_OUT) return MOE_ERR_INVALID_ARG;
  const bool mx = cfg->precision == MOE_MXFP8;
  if (!weight_matches(W13, cfg->precision, E, 2 * F, D) || !weight_matches(W2, cfg->precision, E, D, F))
    return MOE_ERR_INVALID_ARG;
  if (!device_error_word || (reinterpret_cast<uintptr_t>(device_error_word) & 3)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !topk_ids || !topk_scores || !out || !is16(x) || !is16(out)) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * K + 31LL * E > (1LL << 28)) return MOE_ERR_CAPACITY;
  const StaticLayout L = static_layout(T, D, F, E, K, mx);
  if (L.total > kStaticScratchBytes) return MOE_ERR_CAPACITY;

  DeviceSetup* dev = nullptr;
  const moe_status st = setup_device(&dev);
  if (st != MOE_OK) return st;
  uint8_t* S = dev->scratch;
  uint32_t* err = device_error_word;
  RoutingPtrs rp;
  rp.hdr = reinterpret_cast<int*>(S + L.hdr);
  rp.counts = reinterpret_cast<int*>(S + L.counts);
  rp.offsets = reinterpret_cast<int*>(S + L.offsets);
  rp.poffsets = reinterpret_cast<int*>(S + L.poffsets);
  rp.perm = reinterpret_cast<int*>(S + L.perm);
  rp.inv = reinterpret_cast<int*>(S + L.inv);
  rp.blocks = reinterpret_cast<int4*>(S + L.blocks);
  rp.scores = reinterpret_cast<float*>(S + L.scores);
  rp.bstart = reinterpret_cast<int*>(S + L.bstart);
  rp.row_block = reinterpret_cast<int*>(S + L.row_block);
  const int R = static_cast<int>(L.r_cap);
  uint8_t* xrow = S + L.xrow;
  uint8_t* xsf = mx ? S + L.xrow_sf : nullptr;
  uint8_t* h2 = S + L.h2row;
  uint8_t* h2sf = mx ? S + L.h2row_sf : nullptr;
  uint8_t* h3 = S + L.h3;
  const int sms = dev->sms;
  const int debug = (cfg->flags & MOE_DEBUG_CHECKS) ? 1 : 0;

  if (launch_route(topk_ids, topk_scores, T, K, E, R, debug, rp, err, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_gather_rows(mx, false, x, D, K, rp, xrow, xsf, R, sms, stream) != cudaSuccess) return MOE_ERR_CUDA;

  GemmLaunch g1{};
  g1.mx = mx;
  g1.na = 2;
  g1.epi = kEpiSwigluFwd;
  g1.mode = kGroupedM;
  if (!make_tmap(&g1.tmA, W13->data, mx, static_cast<int64_t>(E) * 2 * F, D, 128) ||
      !make_tmap(&g1.tmB, xrow, mx, R, D, 32) ||
      !make_grouped_m_boxes(&g1, W13->data, static_cast<int64_t>(E) * 2 * F, W13->scale, xrow, R, mx, D, F))
    return MOE_ERR_CUDA;
  g1.p.hdr = rp.hdr;
  g1.p.blocks = rp.blocks;
  g1.p.poffsets = rp.poffsets;
  g1.p.E = E;
  g1.p.b_box_rows = 32;
  g1.p.n_tiles = F / 128;
  g1.p.K = D;
  g1.p.a_rows_per_expert = 2 * F;
  g1.p.a_up_offset = F;
  g1.p.sfa = W13->scale;
  g1.p.sfa_ts = D / 128;
  g1.p.sfb = xsf;
  g1.p.sfb_ts = D / 128;
  g1.p.out0 = h2;
  g1.p.out0_pitch = F;
  g1.p.out0_sf = h2sf;
  g1.p.out0_sf_kg = F / 128;
  g1.p.b_cap = static_cast<int>(L.b_cap);
  g1.p.F = F;
  g1.p.swiglu_limit = cfg->swiglu_limit;   // clamped SwiGLU (no clip counters here)
  g1.p.err = err;
  g1.max_tiles = static_cast<int>(L.b_cap * (F / 128));
  if (launch_gemm(g1, sms, stream) != cudaSuccess) return MOE_ERR_CUDA;

  GemmLaunch g2{};
  g2.mx = mx;
  g2.na = pair_tiles(D);
  g2.epi = kEpiStore;
  g2.mode = kGroupedM;
  if (!make_tmap(&g2.tmA, W2->data, mx, static_cast<int64_t>(E) * D, F, 128) ||
      !make_tmap(&g2.tmB, h2, mx, R, F, 32) ||
      !make_grouped_m_boxes(&g2, W2->data, static_cast<int64_t>(E) * D, W2->scale, h2, R, mx, F))
    return MOE_ERR_CUDA;
  g2.p.hdr = rp.hdr;
  g2.p.blocks = rp.blocks;
  g2.p.poffsets = rp.poffsets;
  g2.p.E = E;
  g2.p.b_box_rows = 32;
  g2.p.n_tiles = D / (128 * g2.na);
  g2.p.K = F;
  g2.p.a_rows_per_expert = D;
  g2.p.sfa = W2->scale;
  g2.p.sfa_ts = F / 128;
  g2.p.sfb = h2sf;
  g2.p.sfb_ts = F / 128;
  g2.p.out0 = h3;
  g2.p.out0_pitch = D;
  g2.p.F = F;
  g2.p.err = err;
  g2.max_tiles = static_cast<int>(L.b_cap * g2.p.n_tiles);
  if (launch_gemm(g2, sms, stream) != cudaSuccess) return MOE_ERR_CUDA;

  if (launch_combine(h3, D, K, rp.inv, rp.scores, out, T, (call_flags & MOE_ACCUMULATE_OUT) != 0, sms, stream) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
