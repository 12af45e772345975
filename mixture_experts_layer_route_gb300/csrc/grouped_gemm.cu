// Host side of the grouped GEMMs: TMA tensor maps, kernel variants, launch.
//
// Three variants (token tile BN x pipeline depth), for bf16 (kind::f16) and fp32
// inputs (kind::tf32); with the automatic tile choice each expert is handled
// by the variant its own row count calls for (all three may run in one call):
//   32-token tiles,  9 stages, experts with <= 32 rows (every expert of a batch
//     of <= 64 tokens): the weight stream dominates, so the ring is deep
//     (9 x 16 KB of weights in flight); gated tokens by TMA gather4.
//   128-token tiles, 6 stages, 33..128 rows: still weight-stream heavy, with
//     6 x 16 KB of weights in flight and one token box per stage.
//   256-token tiles, 4 stages, > 128 rows: tensor-core bound, 128 x 256 tiles.
// 128- and 256-token gated tiles read the routed token rows from their
// expert-ordered copy, one TMA box per stage; the down projection always
// loads its h rows that way. CTA pairs share each token tile (multicast) when
// every group has an even number of feature blocks.
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
  const uint32_t es = dtype == MOE_DTYPE_BF16 ? 2 : 4;
  const CUtensorMapDataType dt =
      dtype == MOE_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * es};
  cuuint32_t box[2] = {128u / es, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

constexpr int kMaxExperts = 1024;  // the C ABI's limit on E
// Automatic tile choice by the rows m of each group: 32-token tiles for
// m <= kLightMax, 128-token tiles up to kMediumMax, 256-token tiles beyond
// (thresholds measured on the Qwen3-, Zipf- and DeepSeek-shaped layers). A batch of
// at most kSmallBatch tokens uses 32-token tiles throughout, so it runs one launch
// per GEMM and needs no expert-ordered copy of its rows.
constexpr int kLightMax = 32;
constexpr int kMediumMax = 128;
constexpr int kSmallBatch = 64;

struct AttrCache {
  std::mutex mu;
  // (kernel pointer, device) pairs that already have the smem attribute set.
  const void* fn[64];
  int dev[64];
  int n = 0;
};
AttrCache g_attr;

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

template <typename TIn, bool GATED, int BN, int STAGES, int BMODE, int CL = 1>
cudaError_t launch_variant(const GroupedGemmArgs& a, int num_sms, int E, size_t upper_tiles,
                           cudaStream_t st) {
  using C = GemmCfg<TIn, GATED, BN, STAGES, BMODE, CL>;
  const size_t smem = C::smem_bytes(E);
  auto fn = grouped_gemm_kernel<TIn, GATED, BN, STAGES, BMODE, CL>;
  // Opt in once to what the largest supported expert count needs, so that a
  // later call with more experts than the first still fits.
  cudaError_t e = ensure_smem_attr((const void*)fn, C::smem_bytes(kMaxExperts));
  if (e != cudaSuccess) return e;
  if (CL == 1) {
    size_t grid = (size_t)num_sms;
    if (upper_tiles < grid) grid = upper_tiles;
    if (grid == 0) return cudaSuccess;
    fn<<<(unsigned)grid, C::THREADS, smem, st>>>(a);
    return cudaGetLastError();
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
  cfg.gridDim = dim3((unsigned)(n * CL), 1, 1);
  e = cudaLaunchKernelEx(&cfg, fn, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Upper bound of the tile count of one variant: groups with rows in [m_lo, m_hi].
size_t tile_upper_bound(int T, int k, int E, int BN, int routed_blocks, int shared_blocks,
                        int m_lo, int m_hi) {
  const size_t slots = (size_t)T * k;
  size_t groups = slots / (size_t)(m_lo < 1 ? 1 : m_lo);
  if (groups > (size_t)E) groups = (size_t)E;
  const size_t shared = (shared_blocks > 0 && T >= m_lo && T <= m_hi) ? 1 : 0;
  return (slots / BN + groups) * (size_t)routed_blocks +
         shared * (size_t)((T + BN - 1) / BN) * shared_blocks;
}

struct Range {
  int lo, hi;
};

// Row ranges of the three variants under the automatic choice, or the whole
// range for an explicit tile. Variants whose range cannot be met (every group
// has at most T rows) are not launched.
void variant_ranges(const GemmProblem& p, Range r[3]) {
  const int big = 1 << 30;
  r[0] = r[1] = r[2] = Range{1, 0};  // empty
  switch (p.tile) {
    case MOE_TILE_DECODE: r[0] = Range{1, big}; break;
    case MOE_TILE_MEDIUM: r[1] = Range{1, big}; break;
    case MOE_TILE_PREFILL: r[2] = Range{1, big}; break;
    default:
      if (p.T <= kSmallBatch) {
        r[0] = Range{1, big};
        break;
      }
      r[0] = Range{1, kLightMax};
      r[1] = Range{kLightMax + 1, kMediumMax};
      if (p.T > kMediumMax) r[2] = Range{kMediumMax + 1, big};
  }
}

}  // namespace

bool tensor_map_encoder_available() { return encoder() != nullptr; }

bool gemm_needs_expert_order_copy(const GemmProblem& p) {
  Range r[3];
  variant_ranges(p, r);
  return r[1].lo <= r[1].hi || r[2].lo <= r[2].hi;
}

cudaError_t launch_swiglu_gemm(const GemmProblem& p, const void* x, const void* xg,
                               const int32_t* offsets, const int32_t* gather_idx, const void* Wg,
                               const void* Wu, const void* Wsg, const void* Wsu, void* h, void* hs,
                               int* status, cudaStream_t st) {
  const bool has_s = p.Is > 0;
  const bool bf16 = p.dtype == MOE_DTYPE_BF16;
  // CTA pairs share each token tile when every group has an even number of
  // 64-row feature blocks.
  const bool pair = (p.I / 64) % 2 == 0 && (!has_s || (p.Is / 64) % 2 == 0);
  Range r[3];
  variant_ranges(p, r);
  const int rb = p.I / 64, sb = has_s ? p.Is / 64 : 0;
  for (int v = 0; v < 3; ++v) {
    if (r[v].lo > r[v].hi) continue;
    const int bn = v == 0 ? 32 : (v == 1 ? 128 : 256);
    const bool cl2 = v > 0 && pair;
    GroupedGemmArgs a;
    memset(&a, 0, sizeof(a));
    bool ok = make_tma_map(&a.tmA[0], Wg, p.dtype, (uint64_t)p.E * p.I, p.H, 64) &&
              make_tma_map(&a.tmA[1], Wu, p.dtype, (uint64_t)p.E * p.I, p.H, 64);
    if (ok && has_s)
      ok = make_tma_map(&a.tmA[2], Wsg, p.dtype, p.Is, p.H, 64) &&
           make_tma_map(&a.tmA[3], Wsu, p.dtype, p.Is, p.H, 64);
    if (ok) {
      if (v == 0) {
        ok = make_tma_map(&a.tmB[0], x, p.dtype, p.T, p.H, 1);
        a.tmB[1] = a.tmB[0];
      } else {  // [0]: routed rows in expert order; [1]: x itself for the shared expert
        if (!xg) return cudaErrorInvalidValue;
        const uint32_t box = cl2 ? bn / 2 : bn;
        ok = make_tma_map(&a.tmB[0], xg, p.dtype, (uint64_t)p.T * p.k, p.H, box) &&
             make_tma_map(&a.tmB[1], x, p.dtype, p.T, p.H, box);
      }
    }
    if (!ok) return cudaErrorInvalidValue;
    if (!has_s) {
      a.tmA[2] = a.tmA[0];
      a.tmA[3] = a.tmA[1];
    }
    a.offsets = offsets;
    a.gather_idx = gather_idx;
    a.topk_w = nullptr;
    a.out = h;
    a.out_shared = hs;
    a.status = status;
    a.limit_ns = p.limit_ns;
    a.T = p.T;
    a.k = p.k;
    a.E = p.E;
    a.KP = p.k + (has_s ? 1 : 0);
    a.n_out_routed = p.I;
    a.n_out_shared = has_s ? p.Is : 64;
    a.kdim_routed = p.H;
    a.kdim_shared = p.H;
    a.ld_out_routed = p.I;
    a.ld_out_shared = has_s ? p.Is : 0;
    a.flags = p.flags;
    a.m_lo = r[v].lo;
    a.m_hi = r[v].hi;
    size_t ub = tile_upper_bound(p.T, p.k, p.E, bn, rb, sb, r[v].lo, r[v].hi);
    cudaError_t e;
    if (v == 0)
      e = bf16 ? launch_variant<__nv_bfloat16, true, 32, 9, kGather4>(a, p.num_sms, p.E, ub, st)
               : launch_variant<float, true, 32, 9, kGather4>(a, p.num_sms, p.E, ub, st);
    else if (v == 1)
      e = cl2 ? (bf16 ? launch_variant<__nv_bfloat16, true, 128, 6, kTiled, 2>(a, p.num_sms, p.E,
                                                                              (ub + 1) / 2, st)
                      : launch_variant<float, true, 128, 6, kTiled, 2>(a, p.num_sms, p.E,
                                                                      (ub + 1) / 2, st))
              : (bf16 ? launch_variant<__nv_bfloat16, true, 128, 6, kTiled>(a, p.num_sms, p.E, ub,
                                                                           st)
                      : launch_variant<float, true, 128, 6, kTiled>(a, p.num_sms, p.E, ub, st));
    else
      e = cl2 ? (bf16 ? launch_variant<__nv_bfloat16, true, 256, 4, kTiled, 2>(a, p.num_sms, p.E,
                                                                              (ub + 1) / 2, st)
                      : launch_variant<float, true, 256, 4, kTiled, 2>(a, p.num_sms, p.E,
                                                                      (ub + 1) / 2, st))
              : (bf16 ? launch_variant<__nv_bfloat16, true, 256, 4, kTiled>(a, p.num_sms, p.E, ub,
                                                                           st)
                      : launch_variant<float, true, 256, 4, kTiled>(a, p.num_sms, p.E, ub, st));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_down_gemm(const GemmProblem& p, const void* h, const void* hs,
                             const int32_t* offsets, const int32_t* gather_idx,
                             const float* topk_w, const void* Wd, const void* Wsd, float* Y,
                             int* status, cudaStream_t st) {
  const bool has_s = p.Is > 0;
  const bool bf16 = p.dtype == MOE_DTYPE_BF16;
  const bool pair = (p.H / 128) % 2 == 0;
  Range r[3];
  variant_ranges(p, r);
  const int rb = p.H / 128, sb = has_s ? p.H / 128 : 0;
  for (int v = 0; v < 3; ++v) {
    if (r[v].lo > r[v].hi) continue;
    const int bn = v == 0 ? 32 : (v == 1 ? 128 : 256);
    const bool cl2 = v > 0 && pair;
    const uint32_t box = cl2 ? bn / 2 : bn;  // token box = token tile, or half for CTA pairs
    GroupedGemmArgs a;
    memset(&a, 0, sizeof(a));
    bool ok = make_tma_map(&a.tmA[0], Wd, p.dtype, (uint64_t)p.E * p.H, p.I, 128) &&
              make_tma_map(&a.tmB[0], h, p.dtype, (uint64_t)p.T * p.k, p.I, box);
    if (ok && has_s)
      ok = make_tma_map(&a.tmA[2], Wsd, p.dtype, p.H, p.Is, 128) &&
           make_tma_map(&a.tmB[1], hs, p.dtype, p.T, p.Is, box);
    if (!ok) return cudaErrorInvalidValue;
    if (!has_s) {
      a.tmA[2] = a.tmA[0];
      a.tmB[1] = a.tmB[0];
    }
    a.tmA[1] = a.tmA[0];
    a.tmA[3] = a.tmA[2];
    a.offsets = offsets;
    a.gather_idx = gather_idx;
    a.topk_w = topk_w;
    a.out = Y;
    a.out_shared = nullptr;
    a.status = status;
    a.limit_ns = p.limit_ns;
    a.T = p.T;
    a.k = p.k;
    a.E = p.E;
    a.KP = p.k + (has_s ? 1 : 0);
    a.n_out_routed = p.H;
    a.n_out_shared = p.H;
    a.kdim_routed = p.I;
    a.kdim_shared = has_s ? p.Is : p.I;
    a.ld_out_routed = p.H;
    a.ld_out_shared = p.H;
    a.flags = p.flags;
    a.m_lo = r[v].lo;
    a.m_hi = r[v].hi;
    size_t ub = tile_upper_bound(p.T, p.k, p.E, bn, rb, sb, r[v].lo, r[v].hi);
    cudaError_t e;
    if (v == 0)
      e = bf16 ? launch_variant<__nv_bfloat16, false, 32, 9, kTiled>(a, p.num_sms, p.E, ub, st)
               : launch_variant<float, false, 32, 9, kTiled>(a, p.num_sms, p.E, ub, st);
    else if (v == 1)
      e = cl2 ? (bf16 ? launch_variant<__nv_bfloat16, false, 128, 6, kTiled, 2>(
                            a, p.num_sms, p.E, (ub + 1) / 2, st)
                      : launch_variant<float, false, 128, 6, kTiled, 2>(a, p.num_sms, p.E,
                                                                       (ub + 1) / 2, st))
              : (bf16 ? launch_variant<__nv_bfloat16, false, 128, 6, kTiled>(a, p.num_sms, p.E,
                                                                            ub, st)
                      : launch_variant<float, false, 128, 6, kTiled>(a, p.num_sms, p.E, ub, st));
    else
      e = cl2 ? (bf16 ? launch_variant<__nv_bfloat16, false, 256, 4, kTiled, 2>(
                            a, p.num_sms, p.E, (ub + 1) / 2, st)
                      : launch_variant<float, false, 256, 4, kTiled, 2>(a, p.num_sms, p.E,
                                                                       (ub + 1) / 2, st))
              : (bf16 ? launch_variant<__nv_bfloat16, false, 256, 4, kTiled>(a, p.num_sms, p.E,
                                                                            ub, st)
                      : launch_variant<float, false, 256, 4, kTiled>(a, p.num_sms, p.E, ub, st));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
