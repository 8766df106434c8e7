// Host-side tensor maps of the GEMM operands and outputs (TMA descriptors
// encoded with the driver's cuTensorMapEncodeTiled), shared by the context
// entry points and the allocation-free forward so both launch the GEMMs in
// the same configuration.
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.cuh"

namespace moe {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2D operand map over a row-major [rows, cols] matrix; boxes are
// `row_bytes` (128, 64 or 32) wide with the matching swizzle and `box_rows`
// tall.
bool make_tmap(CUtensorMap* tm, const void* base, bool mx, int64_t rows, int64_t cols, int box_rows,
               int row_bytes) {
  auto fn = encode_fn();
  if (!fn) return false;
  const CUtensorMapDataType dt = mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int esz = mx ? 1 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * esz)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(row_bytes / esz), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : (row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  const CUresult r = fn(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Weight tiles per stage of a grouped-M store GEMM whose output has `n`
// features: two adjacent 128-row tiles share each loaded
// activation box and its scales (half the activation traffic per weight
// byte) when n is a multiple of 256, else one.
int pair_tiles(int64_t n) { return n % 256 == 0 ? 2 : 1; }

// The narrow-box maps a weight-gradient GEMM uses for a short last stage.
bool make_narrow_tmaps(GemmLaunch* g, const void* a, int64_t a_rows, const void* b, int64_t b_rows, bool mx,
                       int64_t cols) {
  return make_tmap(&g->aux[0], a, mx, a_rows, cols, 128, 64) && make_tmap(&g->aux[1], b, mx, b_rows, cols, 128, 64) &&
         make_tmap(&g->aux[2], a, mx, a_rows, cols, 128, 32) && make_tmap(&g->aux[3], b, mx, b_rows, cols, 128, 32);
}

// A tensor map of any rank (dims / box innermost first, byte strides of
// dims 1..rank-1), no interleave.
bool make_tmap_nd(CUtensorMap* tm, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
                  const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(tm, dt, rank, const_cast<void*>(base), const_cast<cuuint64_t*>(dims), const_cast<cuuint64_t*>(strides),
            const_cast<cuuint32_t*>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The larger boxes a grouped-M GEMM loads with (fewer copies per stage for
// the producer thread to issue):
//  * both A tiles of a stage in one copy: a 256-row box when they are
//    adjacent (store GEMMs with two tiles per stage), a 3D box over
//    [2E halves][F rows][K] when they are W13's gate and up halves
//    (`halves_f` = F), and likewise their two MXFP8 scale atoms, read as
//    [row tiles][K/128][128 words] (adjacent) or [2E][F/128][K/128][128]
//    (halves) from `a_sf`;
//  * a full 128-row routing block of B in one box.
// Over row-block pairs (kGroupedMP) the SwiGLU forward's one A tile is the
// same 3D box 64 rows high: 64 gate rows, then the up rows of the same
// features.
//
// On CTA pairs (kGroupedMC) a stage is two 128-byte K-chunks, and each box
// covers both: the K axis is split into [chunks][128 bytes] (the chunk axis
// outermost in the box), so a box lands as [chunk][rows][128 B], one 128-row
// (or 2 x 64-row) tile per chunk.  aux[0]: A (W13: [chunks]
// [gate, up][64 rows]; W2: [chunks][128 rows]); aux[1]: B, one routing block
// ([chunks][128 rows]); aux[2] (W13): both chunks' atoms of the gate and up
// halves.
bool make_grouped_m_boxes(GemmLaunch* g, const void* a, int64_t a_rows, const void* a_sf, const void* b,
                          int64_t b_rows, bool mx, int64_t cols, int64_t halves_f) {
  const int esz = mx ? 1 : 2;
  const CUtensorMapDataType dt = mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint64_t ks = static_cast<cuuint64_t>(cols / 128), atom = 512;
  if (g->mode == kGroupedMC) {
    const cuuint64_t w = static_cast<cuuint64_t>(128 / esz);             // elements per chunk
    if (cols % (2 * w) != 0) return false;
    const cuuint64_t nch = static_cast<cuuint64_t>(cols) / w;           // chunks along K
    const cuuint64_t rb = static_cast<cuuint64_t>(cols) * esz;          // row pitch in bytes
    if (g->epi == kEpiSwigluFwd) {
      if (halves_f <= 0 || halves_f % 128 != 0) return false;
      const cuuint64_t hf = static_cast<cuuint64_t>(halves_f);
      const cuuint64_t d[4] = {w, hf, static_cast<cuuint64_t>(a_rows) / hf, nch};
      const cuuint64_t st[3] = {rb, hf * rb, 128};
      const cuuint32_t bx[4] = {static_cast<cuuint32_t>(w), 64, 2, 2};
      if (!make_tmap_nd(&g->aux[0], dt, 4, a, d, st, bx, CU_TENSOR_MAP_SWIZZLE_128B)) return false;
      if (mx) {
        const cuuint64_t ft = hf / 128;
        const cuuint64_t d4[4] = {128, ks, ft, static_cast<cuuint64_t>(a_rows) / hf};
        const cuuint64_t st4[3] = {atom, ks * atom, ft * ks * atom};
        const cuuint32_t bx4[4] = {128, 2, 1, 2};
        if (!make_tmap_nd(&g->aux[2], CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, a_sf, d4, st4, bx4,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
          return false;
      }
    } else {
      const cuuint64_t d[3] = {w, static_cast<cuuint64_t>(a_rows), nch};
      const cuuint64_t st[2] = {rb, 128};
      const cuuint32_t bx[3] = {static_cast<cuuint32_t>(w), 128, 2};
      if (!make_tmap_nd(&g->aux[0], dt, 3, a, d, st, bx, CU_TENSOR_MAP_SWIZZLE_128B)) return false;
    }
    const cuuint64_t d[3] = {w, static_cast<cuuint64_t>(b_rows), nch};
    const cuuint64_t st[2] = {rb, 128};
    const cuuint32_t bx[3] = {static_cast<cuuint32_t>(w), 128, 2};
    if (!make_tmap_nd(&g->aux[1], dt, 3, b, d, st, bx, CU_TENSOR_MAP_SWIZZLE_128B)) return false;
    g->p.a_pair_box = 0;
    g->p.b_full_box = 0;
    return true;
  }
  if (g->na == 2 && g->epi == kEpiStore) {
    if (!make_tmap(&g->aux[0], a, mx, a_rows, cols, 256)) return false;
    if (mx) {
      const cuuint64_t d[3] = {128, ks, static_cast<cuuint64_t>(a_rows / 128)};
      const cuuint64_t st[2] = {atom, ks * atom};
      const cuuint32_t bx[3] = {128, 1, 2};
      if (!make_tmap_nd(&g->aux[2], CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, a_sf, d, st, bx, CU_TENSOR_MAP_SWIZZLE_NONE))
        return false;
    }
    g->p.a_pair_box = 1;
  } else if ((g->na == 2 || g->mode == kGroupedMP) && g->epi == kEpiSwigluFwd && halves_f > 0 &&
             halves_f % 128 == 0) {
    const cuuint64_t d[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(halves_f),
                             static_cast<cuuint64_t>(a_rows / halves_f)};
    const cuuint64_t st[2] = {static_cast<cuuint64_t>(cols * esz), static_cast<cuuint64_t>(halves_f * cols * esz)};
    const cuuint32_t bx[3] = {static_cast<cuuint32_t>(128 / esz), g->na == 1 ? 64u : 128u, 2};
    if (!make_tmap_nd(&g->aux[0], dt, 3, a, d, st, bx, CU_TENSOR_MAP_SWIZZLE_128B)) return false;
    if (mx) {
      const cuuint64_t ft = static_cast<cuuint64_t>(halves_f / 128);
      const cuuint64_t d4[4] = {128, ks, ft, static_cast<cuuint64_t>(a_rows / halves_f)};
      const cuuint64_t st4[3] = {atom, ks * atom, ft * ks * atom};
      const cuuint32_t bx4[4] = {128, 1, 1, 2};
      if (!make_tmap_nd(&g->aux[2], CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, a_sf, d4, st4, bx4,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
        return false;
    }
    g->p.a_pair_box = 2;
  }
  if (!make_tmap(&g->aux[1], b, mx, b_rows, cols, 128)) return false;
  g->p.b_full_box = 1;
  return true;
}

// Output map of a weight gradient [rows, cols]: boxes of 128 bytes (64 BF16
// or 32 FP32 columns) x 128 rows in the 128-byte swizzle the epilogue stages.
bool make_out_tmap(CUtensorMap* tm, void* base, int64_t rows, int64_t cols, bool fp32) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int esz = fp32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * esz)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz), 128};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace moe
