// Host side of the grouped GEMMs: TMA tensor maps, kernel variants, launch.
//
// One launch per GEMM, for bf16 (kind::f16) and fp32 inputs (kind::tf32):
//   decode-sized batches (T <= 64, or MOE_TILE_DECODE): 32-token tiles, 9
//     stages of 16 KB of weights; the gated GEMM gathers its token rows with
//     TMA gather4, so no expert-ordered copy of x is made;
//   otherwise: token tiles of up to 256 rows on CTA pairs (cta_group::2
//     MMAs, M = 256, 3 stages of two 128-byte K boxes, 64 KB per SM;
//     MOE_TILE_MEDIUM: 128 rows, 4 stages of 48 KB; one box per stage, twice
//     the stages, when a contraction length is not a multiple of two boxes),
//     every expert in the same launch, heaviest experts first; the gated GEMM reads
//     the routed rows from their expert-ordered copy and each tile loads the
//     smallest token box (128, 64 or 16 rows per CTA) that covers it. Groups
//     with an odd number of feature blocks fall back to single-CTA tiles.
#include <mutex>

#include <cudaTypedefs.h>

#include "grouped_gemm.cuh"
#include "kernels.h"

namespace moe {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// cuTensorMapEncodeTiled, looked up once through the runtime (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}
}  // namespace

// 2-D row-major matrix [rows][cols] of `es`-byte elements; box = 128 bytes of
// columns x box_rows rows, 128-byte swizzle.
bool make_tma_map(CUtensorMap* m, const void* base, int dtype, uint64_t rows, uint64_t cols,
                  uint32_t box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  const uint32_t es = dtype == MOE_DTYPE_BF16 ? 2 : (dtype == MOE_DTYPE_E4M3 ? 1 : 4);
  const CUtensorMapDataType dt = dtype == MOE_DTYPE_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : dtype == MOE_DTYPE_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * es};
  cuuint32_t box[2] = {128u / es, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D uint8 matrix [rows][cols] (E4M3 codes) with boxes of 64 bytes of columns
// x box_rows rows, 64-byte swizzle (16-byte chunk c of a box row r lands at
// chunk position c ^ ((r >> 1) & 3)).
bool make_code_map64(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows) {
  auto enc = encoder();
  if (!enc || cols % 16 != 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D uint8 matrix [rows][cols] (cols a multiple of 16) whose box is box_cols
// bytes (whole rows when 0; a multiple of 16, at most 256) x box_rows rows, no
// swizzle. The MX scale rows.
bool make_scale_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t cols,
                    uint32_t box_rows, uint32_t box_cols) {
  auto enc = encoder();
  if (box_cols == 0) box_cols = cols;
  if (!enc || cols % 16 != 0 || box_cols % 16 != 0 || box_cols > 256 || box_cols > cols)
    return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

constexpr int kMaxExperts = 1024;  // the C ABI's limit on E
// A batch of at most kSmallBatch tokens runs the 32-token gather4 kernel: its
// experts hold a few rows each, and its rows need no expert-ordered copy.
constexpr int kSmallBatch = 64;

struct AttrCache {
  std::mutex mu;
  // (kernel pointer, device) pairs that already have the smem attribute set.
  const void* fn[64];
  int dev[64];
  int n = 0;
};
AttrCache g_attr;

}  // namespace

cudaError_t ensure_smem_attr(const void* fn, size_t smem) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_attr.mu);
  for (int i = 0; i < g_attr.n; ++i)
    if (g_attr.fn[i] == fn && g_attr.dev[i] == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess && g_attr.n < 64) {
    g_attr.fn[g_attr.n] = fn;
    g_attr.dev[g_attr.n] = dev;
    ++g_attr.n;
  }
  return e;
}

namespace {

template <typename TIn, bool GATED, int BN, int STAGES, int BMODE, int CL = 1, int NBX = 1>
cudaError_t launch_variant(const GroupedGemmArgs& a, int num_sms, int E, size_t upper_tiles,
                           cudaStream_t st) {
  using C = GemmCfg<TIn, GATED, BN, STAGES, BMODE, CL, NBX>;
  const size_t smem = C::smem_bytes(E);
  auto fn = grouped_gemm_kernel<TIn, GATED, BN, STAGES, BMODE, CL, NBX>;
  // Opt in once to what the largest supported expert count needs, so that a
  // later call with more experts than the first still fits.
  cudaError_t e = ensure_smem_attr((const void*)fn, C::smem_bytes(kMaxExperts));
  if (e != cudaSuccess) return e;
  if (CL == 1) {
    size_t grid = (size_t)num_sms;
    if (upper_tiles < grid) grid = upper_tiles;
    if (grid == 0) return cudaSuccess;
    return launch_chained(fn, dim3((unsigned)grid), dim3(C::THREADS), smem, st, 1, a);
  }
  // Persistent grid of as many CTA pairs as can be resident at once; upper_tiles
  // counts pair units here.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((unsigned)(num_sms / CL * CL), 1, 1);
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, (const void*)fn, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  size_t n = (size_t)clusters;
  if (upper_tiles < n) n = upper_tiles;
  if (n == 0) return cudaSuccess;
  return launch_chained(fn, dim3((unsigned)(n * CL)), dim3(C::THREADS), smem, st, CL, a);
}

}  // namespace

// Upper bound of the unit count of one launch: T*k routed rows in at most
// min(E, T*k) groups of ceil(m / tile_n) token tiles each, plus the shared
// expert's T rows.
size_t unit_upper_bound(int T, int k, int E, int tile_n, int routed_blocks, int shared_blocks) {
  const size_t slots = (size_t)T * k;
  const size_t groups = slots < (size_t)E ? slots : (size_t)E;
  return (slots / tile_n + groups) * (size_t)routed_blocks +
         (size_t)((T + tile_n - 1) / tile_n) * shared_blocks;
}

namespace {

// One launch per GEMM: the 32-token gather4 kernel for decode-sized batches
// (or when forced), otherwise the tiled kernel with token tiles of tile_n rows.
bool use_decode_kernel(const GemmProblem& p) {
  return p.tile == MOE_TILE_DECODE || (p.tile == MOE_TILE_AUTO && p.T <= kSmallBatch);
}

// Token tile of the tiled kernel: 256 (3 stages of 64 KB per SM), or 128 (4
// stages of 48 KB) when forced. 128-token tiles measured slower on every
// layer shape: a 256 x 128 pair MMA step is fed at ~94 B/clk per SM, and an
// expert of 129..256 rows then streams its weights to the SMs twice.
int tiled_tile_n(const GemmProblem& p) { return p.tile == MOE_TILE_MEDIUM ? 128 : 256; }

}  // namespace

// Tensor maps of a tiled token operand [rows][cols]: boxes of b_rows, box1 and
// 16 rows (GemmCfg::B_ROWS, BOX1).
bool make_b_maps(CUtensorMap* m, const void* base, int dtype, uint64_t rows, uint64_t cols,
                 uint32_t b_rows, uint32_t box1) {
  return make_tma_map(&m[0], base, dtype, rows, cols, b_rows) &&
         make_tma_map(&m[1], base, dtype, rows, cols, box1) &&
         make_tma_map(&m[2], base, dtype, rows, cols, 16);
}

namespace {

void fill_common(GroupedGemmArgs& a, const GemmProblem& p, const int32_t* offsets,
                 const int32_t* gather_idx, int* status, int tile_n) {
  a.offsets = offsets;
  a.gather_idx = gather_idx;
  a.status = status;
  a.limit_ns = p.limit_ns;
  a.T = p.T;
  a.k = p.k;
  a.E = p.E;
  a.KP = p.k + (p.Is > 0 ? 1 : 0);
  a.flags = p.flags;
  a.m_lo = 1;
  a.m_hi = 1 << 30;
  a.tile_n = tile_n;
}

// Pre-wait weight prefetch (GroupedGemmArgs::pf_first): decode-sized launches
// without a shared expert, with at least 4 routed slots per expert on average
// (an expert then holds no rows with probability ~e^-4 under uniform routing,
// and none holds more than a 32-row tile, so the schedule is index order).
bool prefetch_first_units(const GemmProblem& p, bool dec) {
  return dec && p.Is == 0 && (int64_t)p.T * p.k >= 4 * (int64_t)p.E;
}

// CTA pairs take two 128-byte K boxes per stage (the MMA issuer then waits and
// commits once per eight MMAs) when every contraction length is a multiple
// of two boxes.
template <typename TIn>
bool two_box_stages(const GroupedGemmArgs& a) {
  const int kb2 = 256 / (int)sizeof(TIn);
  return a.kdim_routed % kb2 == 0 && a.kdim_shared % kb2 == 0;
}

template <typename TIn>
cudaError_t launch_gated(const GroupedGemmArgs& a, const GemmProblem& p, bool dec, bool pair,
                         int tile_n, size_t ub, cudaStream_t st) {
  if (dec) return launch_variant<TIn, true, 32, 9, kGather4>(a, p.num_sms, p.E, ub, st);
  const size_t pu = (ub + 1) / 2;
  const bool two = two_box_stages<TIn>(a);
  if (pair && tile_n == 128)
    return two ? launch_variant<TIn, true, 128, 4, kTiled, 2, 2>(a, p.num_sms, p.E, pu, st)
               : launch_variant<TIn, true, 128, 8, kTiled, 2>(a, p.num_sms, p.E, pu, st);
  if (pair)
    return two ? launch_variant<TIn, true, 256, 3, kTiled, 2, 2>(a, p.num_sms, p.E, pu, st)
               : launch_variant<TIn, true, 256, 6, kTiled, 2>(a, p.num_sms, p.E, pu, st);
  return launch_variant<TIn, true, 256, 4, kTiled>(a, p.num_sms, p.E, ub, st);
}

template <typename TIn>
cudaError_t launch_down(const GroupedGemmArgs& a, const GemmProblem& p, bool dec, bool pair,
                        int tile_n, size_t ub, cudaStream_t st) {
  if (dec) return launch_variant<TIn, false, 32, 9, kTiled>(a, p.num_sms, p.E, ub, st);
  const size_t pu = (ub + 1) / 2;
  const bool two = two_box_stages<TIn>(a);
  if (pair && tile_n == 128)
    return two ? launch_variant<TIn, false, 128, 4, kTiled, 2, 2>(a, p.num_sms, p.E, pu, st)
               : launch_variant<TIn, false, 128, 8, kTiled, 2>(a, p.num_sms, p.E, pu, st);
  if (pair)
    return two ? launch_variant<TIn, false, 256, 3, kTiled, 2, 2>(a, p.num_sms, p.E, pu, st)
               : launch_variant<TIn, false, 256, 6, kTiled, 2>(a, p.num_sms, p.E, pu, st);
  return launch_variant<TIn, false, 256, 4, kTiled>(a, p.num_sms, p.E, ub, st);
}

}  // namespace

bool tensor_map_encoder_available() { return encoder() != nullptr; }

bool gemm_uses_decode_tiles(const GemmProblem& p) { return use_decode_kernel(p); }

bool gemm_needs_expert_order_copy(const GemmProblem& p) { return !use_decode_kernel(p); }

// Arguments of the gate/up GEMM (see kernels.h); false if a tensor map
// cannot be made.
bool prepare_swiglu_gemm(GroupedGemmArgs& a, const GemmProblem& p, const void* x, const void* xg,
                         const int32_t* offsets, const int32_t* gather_idx, const void* Wg,
                         const void* Wu, const void* Wsg, const void* Wsu, void* h, void* hs,
                         int* status, const GemmScales* sc) {
  const bool has_s = p.Is > 0;
  const bool dec = use_decode_kernel(p);
  // CTA pairs when every group has an even number of 64-row feature blocks.
  const bool pair = !dec && (p.I / 64) % 2 == 0 && (!has_s || (p.Is / 64) % 2 == 0);
  const int tile_n = dec ? 32 : tiled_tile_n(p);
  memset(&a, 0, sizeof(a));
  bool ok = make_tma_map(&a.tmA[0], Wg, p.dtype, (uint64_t)p.E * p.I, p.H, 64) &&
            make_tma_map(&a.tmA[1], Wu, p.dtype, (uint64_t)p.E * p.I, p.H, 64);
  if (ok && has_s)
    ok = make_tma_map(&a.tmA[2], Wsg, p.dtype, p.Is, p.H, 64) &&
         make_tma_map(&a.tmA[3], Wsu, p.dtype, p.Is, p.H, 64);
  if (ok) {
    if (dec) {
      ok = make_tma_map(&a.tmB[0], x, p.dtype, p.T, p.H, 1);
    } else {  // [0..2]: routed rows in expert order; [3..5]: x itself for the shared expert
      if (!xg) return false;
      const uint32_t br = pair ? tile_n / 2 : 256, b1 = br / 2;
      ok = make_b_maps(&a.tmB[0], xg, p.dtype, (uint64_t)p.T * p.k, p.H, br, b1) &&
           make_b_maps(&a.tmB[3], x, p.dtype, p.T, p.H, br, b1);
    }
  }
  if (!ok) return false;
  if (!has_s) {
    a.tmA[2] = a.tmA[0];
    a.tmA[3] = a.tmA[1];
  }
  fill_common(a, p, offsets, gather_idx, status, tile_n);
  a.pf_first = prefetch_first_units(p, dec) ? 1 : 0;
  a.pf_base[0] = Wg;
  a.pf_base[1] = Wu;
  a.topk_w = nullptr;
  if (sc) {
    for (int i = 0; i < 4; ++i) a.sA[i] = sc->a[i];
    for (int i = 0; i < 2; ++i) a.sB[i] = sc->b[i];
  }
  a.out = h;
  a.out_shared = hs;
  a.n_out_routed = p.I;
  a.n_out_shared = has_s ? p.Is : 64;
  a.kdim_routed = p.H;
  a.kdim_shared = p.H;
  a.ld_out_routed = p.I;
  a.ld_out_shared = has_s ? p.Is : 0;
  return true;
}

cudaError_t launch_swiglu_gemm(const GemmProblem& p, const void* x, const void* xg,
                               const int32_t* offsets, const int32_t* gather_idx, const void* Wg,
                               const void* Wu, const void* Wsg, const void* Wsu, void* h, void* hs,
                               int* status, cudaStream_t st, const GemmScales* sc) {
  GroupedGemmArgs a;
  if (!prepare_swiglu_gemm(a, p, x, xg, offsets, gather_idx, Wg, Wu, Wsg, Wsu, h, hs, status, sc))
    return cudaErrorInvalidValue;
  const bool has_s = p.Is > 0;
  const bool dec = use_decode_kernel(p);
  const bool pair = !dec && (p.I / 64) % 2 == 0 && (!has_s || (p.Is / 64) % 2 == 0);
  const int tile_n = a.tile_n;
  const int rb = p.I / 64, sb = has_s ? p.Is / 64 : 0;
  const size_t ub = unit_upper_bound(p.T, p.k, p.E, tile_n, rb, sb);
  switch (p.dtype) {
    case MOE_DTYPE_BF16:
      return launch_gated<__nv_bfloat16>(a, p, dec, pair, tile_n, ub, st);
    case MOE_DTYPE_E4M3:
      return launch_gated<uint8_t>(a, p, dec, pair, tile_n, ub, st);
    default:
      return launch_gated<float>(a, p, dec, pair, tile_n, ub, st);
  }
}

// Arguments of the down GEMM (see kernels.h); false if a tensor map cannot be
// made.
bool prepare_down_gemm(GroupedGemmArgs& a, const GemmProblem& p, const void* h, const void* hs,
                       const int32_t* offsets, const int32_t* gather_idx, const float* topk_w,
                       const void* Wd, const void* Wsd, float* Y, int* status,
                       const GemmScales* sc) {
  const bool has_s = p.Is > 0;
  const bool dec = use_decode_kernel(p);
  const bool pair = !dec && (p.H / 128) % 2 == 0;
  const int tile_n = dec ? 32 : tiled_tile_n(p);
  // Token boxes: B_ROWS and BOX1 of the variant launched (decode: 32 and 16).
  const uint32_t br = dec ? 32 : (pair ? tile_n / 2 : 256), b1 = br / 2 < 16 ? 16 : br / 2;
  memset(&a, 0, sizeof(a));
  bool ok = make_tma_map(&a.tmA[0], Wd, p.dtype, (uint64_t)p.E * p.H, p.I, 128) &&
            make_b_maps(&a.tmB[0], h, p.dtype, (uint64_t)p.T * p.k, p.I, br, b1);
  if (ok && has_s)
    ok = make_tma_map(&a.tmA[2], Wsd, p.dtype, p.H, p.Is, 128) &&
         make_b_maps(&a.tmB[3], hs, p.dtype, p.T, p.Is, br, b1);
  if (!ok) return false;
  if (!has_s) {
    a.tmA[2] = a.tmA[0];
    for (int i = 0; i < 3; ++i) a.tmB[3 + i] = a.tmB[i];
  }
  a.tmA[1] = a.tmA[0];
  a.tmA[3] = a.tmA[2];
  fill_common(a, p, offsets, gather_idx, status, tile_n);
  a.pf_first = prefetch_first_units(p, dec) ? 1 : 0;
  a.pf_base[0] = Wd;
  a.pf_base[1] = Wd;
  a.topk_w = topk_w;
  if (sc) {
    for (int i = 0; i < 4; ++i) a.sA[i] = sc->a[i];
    for (int i = 0; i < 2; ++i) a.sB[i] = sc->b[i];
  }
  a.out = Y;
  a.out_shared = nullptr;
  a.n_out_routed = p.H;
  a.n_out_shared = p.H;
  a.kdim_routed = p.I;
  a.kdim_shared = has_s ? p.Is : p.I;
  a.ld_out_routed = p.H;
  a.ld_out_shared = p.H;
  return true;
}

cudaError_t launch_down_gemm(const GemmProblem& p, const void* h, const void* hs,
                             const int32_t* offsets, const int32_t* gather_idx,
                             const float* topk_w, const void* Wd, const void* Wsd, float* Y,
                             int* status, cudaStream_t st, const GemmScales* sc) {
  GroupedGemmArgs a;
  if (!prepare_down_gemm(a, p, h, hs, offsets, gather_idx, topk_w, Wd, Wsd, Y, status, sc))
    return cudaErrorInvalidValue;
  const bool has_s = p.Is > 0;
  const bool dec = use_decode_kernel(p);
  const bool pair = !dec && (p.H / 128) % 2 == 0;
  const int tile_n = a.tile_n;
  const int rb = p.H / 128, sb = has_s ? p.H / 128 : 0;
  const size_t ub = unit_upper_bound(p.T, p.k, p.E, tile_n, rb, sb);
  switch (p.dtype) {
    case MOE_DTYPE_BF16:
      return launch_down<__nv_bfloat16>(a, p, dec, pair, tile_n, ub, st);
    case MOE_DTYPE_E4M3:
      return launch_down<uint8_t>(a, p, dec, pair, tile_n, ub, st);
    default:
      return launch_down<float>(a, p, dec, pair, tile_n, ub, st);
  }
}

}  // namespace moe
