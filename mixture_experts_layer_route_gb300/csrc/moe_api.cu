// C ABI entry points: argument validation, workspace layout, kernel sequence.
// Every launch goes to the caller's stream; nothing here synchronises except
// moe_get_device_status().
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "moe_api.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// NVTX range around host-side work (an entry point, one launch): a profiler
// that records NVTX shows each stage's launch under its name; without one
// the calls return at once.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr size_t kAlign = 256;
constexpr size_t kHeader = 256;  // status word + reserved
// Header words: the status word at int 0; the single-launch decode kernel's
// grid-barrier counter at int 16 (its own 64-byte line). moe_forward and
// moe_forward_single_launch clear the first kHeaderClear bytes.
constexpr int kGridCounter = 16;
constexpr size_t kHeaderClear = 128;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t pscratch, logits, partials, ids, w, offsets, gather, slotpos, xg, h, hs, Y, units, fpart,
      total;
  // E4M3 layers only: quantized token rows and scales, quantized h rows and
  // scales (routed and shared); 0 otherwise.
  size_t xq, sx, hq, sh, hsq, shs;
  size_t xm;  // MXFP8 layers only: quantized token rows (bf16 values); 0 otherwise
  // MXFP8 layers on the decode-sized kernels: token codes and scale rows
  // (xq above holds the codes), their expert-ordered copies (xg holds the
  // codes), and the scale rows of h and h_shared (h, hs hold the codes).
  size_t xs, xgs, hsc, hss;
  bool mx_dec;
  int S;  // router split count
};

// Number of SMs used to size the router split; a fixed value keeps the
// workspace size independent of the device queried.
constexpr int kRouterSplitSms = 152;

// 128/256-token tiles read the routed token rows from an expert-ordered copy;
// they can run unless every expert is forced to, or bound to, 32-token tiles.
bool needs_copy(const moe_problem& p) {
  if (p.tile == MOE_TILE_DECODE) return false;
  if (p.tile == MOE_TILE_AUTO) return p.T > 64;
  return true;
}

// Bytes of one element of the expert GEMM operands (E4M3 codes: 1).
// MXFP8 layers: 2 (their token operands are bf16 rows holding MXFP8 values).
size_t elem_bytes(int dtype) {
  return (dtype == MOE_DTYPE_BF16 || dtype == MOE_DTYPE_MXFP8) ? 2
                                                               : (dtype == MOE_DTYPE_E4M3 ? 1 : 4);
}
// Dtype of the activations (x, W_router, h, y): bf16 for E4M3 and MXFP8 layers.
int act_dtype(int dtype) {
  return (dtype == MOE_DTYPE_E4M3 || dtype == MOE_DTYPE_MXFP8) ? MOE_DTYPE_BF16 : dtype;
}

// MXFP8 problems with decode-sized token tiles run the E4M3-MMA kernels
// (grouped_gemm_mx.cu), whose token operands are codes with scale rows.
bool mx_decode_kernels(const moe_problem& p) {
  return p.tile == MOE_TILE_DECODE || (p.tile == MOE_TILE_AUTO && p.T <= 64);
}

Layout layout_of(const moe_problem& p) {
  Layout L;
  const size_t es = elem_bytes(p.dtype);
  const size_t T = (size_t)p.T, E = (size_t)p.E, k = (size_t)p.k;
  const size_t KP = k + (p.I_shared > 0 ? 1 : 0);
  const bool f8 = p.dtype == MOE_DTYPE_E4M3;
  const bool mx = p.dtype == MOE_DTYPE_MXFP8;
  const size_t as = elem_bytes(act_dtype(p.dtype));
  L.S = router_split_count(act_dtype(p.dtype), p.T, p.H, p.E, kRouterSplitSms);
  size_t off = kHeader;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  // First after the header: moe_permute (which has no problem struct) finds
  // its per-chunk counts here from T, E and k alone.
  L.pscratch = take(permute_scratch_bytes(p.T, p.E, p.k));
  L.logits = take(T * E * 4);
  L.partials = L.S > 1 ? take((size_t)L.S * T * E * 4) : L.logits;
  L.ids = take(T * k * 4);
  L.w = take(T * k * 4);
  L.offsets = take((E + 2) * 4);
  L.gather = take(T * k * 4);
  L.slotpos = take(T * k * 4);
  // Prefill-sized tiles read the routed token rows from an expert-ordered copy.
  L.xq = f8 ? take(T * (size_t)p.H) : 0;
  L.sx = f8 ? take(T * 4) : 0;
  // MXFP8 layers: the quantized token rows (bf16 values, or E4M3 codes and
  // scale rows for the decode-sized kernels), and always their expert-ordered
  // copy (both MXFP8 GEMMs read tiled token rows).
  L.mx_dec = mx && mx_decode_kernels(p);
  L.xm = mx && !L.mx_dec ? take(T * (size_t)p.H * 2) : 0;
  if (L.mx_dec) {
    const size_t skH = (size_t)moe_mx_scale_cols(p.H);
    L.xq = take(T * (size_t)p.H);
    L.xs = take(T * skH);
    L.xgs = take(T * k * skH);
    L.hsc = take(T * k * (size_t)moe_mx_scale_cols(p.I));
    L.hss = p.I_shared > 0 ? take(T * (size_t)moe_mx_scale_cols(p.I_shared)) : 0;
  } else {
    L.xs = L.xgs = L.hsc = L.hss = 0;
  }
  L.xg = (needs_copy(p) || mx) ? take(T * k * (size_t)p.H * es) : 0;
  L.h = take(T * k * (size_t)p.I * as);
  L.hs = p.I_shared > 0 ? take(T * (size_t)p.I_shared * as) : 0;
  L.hq = f8 ? take(T * k * (size_t)p.I) : 0;
  L.sh = f8 ? take(T * k * 4) : 0;
  L.hsq = f8 && p.I_shared > 0 ? take(T * (size_t)p.I_shared) : 0;
  L.shs = f8 && p.I_shared > 0 ? take(T * 4) : 0;
  L.Y = take(T * KP * (size_t)p.H * 4);
  // Single-launch decode kernel: per-group counts of finished gate/up units.
  L.units = take((E + 2) * 4);
  // ... and its router partial sums (at most 8 slices of H), for decode-sized
  // batches only.
  L.fpart = T <= 64 ? take(8 * T * E * 4) : 0;
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Group-limited routing parameters (n_group <= 1: plain top-k, always valid).
bool groups_valid(int64_t E, int64_t k, int64_t n_group, int64_t topk_group) {
  if (n_group <= 1) return true;
  if (n_group > 32 || E % n_group != 0) return false;
  if (topk_group < 1 || topk_group > n_group) return false;
  return k <= topk_group * (E / n_group);
}

int* status_ptr(void* ws) { return reinterpret_cast<int*>(ws); }

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(reinterpret_cast<uint8_t*>(ws) + off);
}

moe_status check_ws(const void* ws, size_t have, size_t need) {
  if (!ws || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  if (have < need) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

std::mutex g_sm_mu;
int g_sm_count[64] = {0};

}  // namespace

// ---- shared with the other entry points of the library (declared in kernels.h)

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lk(g_sm_mu);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return 148;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

// Host-side validation of a problem, before any launch. allow_quantized: the
// entry points that take quantized weights (workspace queries,
// moe_forward_fp8 and moe_forward_mx); the bf16/fp32 sub-calls reject those
// dtypes.
moe_status check_problem(const moe_problem* pb, bool allow_quantized) {
  if (!pb) return MOE_ERR_INVALID_ARG;
  const moe_problem& p = *pb;
  if (p.T < 0 || p.H <= 0 || p.E <= 0 || p.k <= 0 || p.I <= 0 || p.I_shared < 0)
    return MOE_ERR_INVALID_ARG;
  if (p.k > p.E || p.k > 32 || p.E > 1024) return MOE_ERR_INVALID_ARG;
  if (p.H % 128 != 0 || p.I % 64 != 0 || p.I_shared % 64 != 0) return MOE_ERR_INVALID_ARG;
  const bool quantized = p.dtype == MOE_DTYPE_E4M3 || p.dtype == MOE_DTYPE_MXFP8;
  if (p.dtype != MOE_DTYPE_BF16 && p.dtype != MOE_DTYPE_F32 && !(allow_quantized && quantized))
    return MOE_ERR_INVALID_ARG;
  // E4M3 and MXFP8 GEMMs take 128 elements of K per stage.
  if (quantized && (p.I % 128 != 0 || p.I_shared % 128 != 0)) return MOE_ERR_INVALID_ARG;
  // An MXFP8 weight row's scales (one byte per 32 elements) are loaded as one
  // box of at most 256 bytes.
  if (p.dtype == MOE_DTYPE_MXFP8 && (p.H > 8192 || p.I > 8192 || p.I_shared > 8192))
    return MOE_ERR_UNSUPPORTED;
  if (p.tile < MOE_TILE_AUTO || p.tile > MOE_TILE_MEDIUM) return MOE_ERR_INVALID_ARG;
  if (p.renorm != 0 && p.renorm != 1) return MOE_ERR_INVALID_ARG;
  if (p.out_f32 != 0 && p.out_f32 != 1) return MOE_ERR_INVALID_ARG;
  if (!groups_valid(p.E, p.k, p.n_group, p.topk_group)) return MOE_ERR_INVALID_ARG;
  const int64_t lim = (int64_t)1 << 30;
  if (p.T * (p.k + 1) >= lim || p.H >= lim || p.I >= lim || p.E * p.I >= lim ||
      p.E * p.H >= lim)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

GemmProblem gemm_problem(const moe_problem& p) {
  GemmProblem g;
  g.dtype = p.dtype;
  g.tile = p.tile;
  g.T = (int)p.T;
  g.H = (int)p.H;
  g.E = (int)p.E;
  g.k = (int)p.k;
  g.I = (int)p.I;
  g.Is = (int)p.I_shared;
  g.flags = p.flags;
  g.limit_ns = (unsigned long long)(p.wait_limit_us ? p.wait_limit_us : 1000000u) * 1000ull;
  g.num_sms = sm_count();
  return g;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status moe_workspace_size(const moe_problem* pb, size_t* bytes) {
  moe_status s = check_problem(pb, true);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = layout_of(*pb).total;
  return MOE_OK;
}

moe_status moe_get_workspace_layout(const moe_problem* pb, moe_workspace_layout* out) {
  moe_status s = check_problem(pb, true);
  if (s != MOE_OK) return s;
  if (!out) return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(*pb);
  out->logits = (int64_t)L.logits;
  out->topk_ids = (int64_t)L.ids;
  out->topk_w = (int64_t)L.w;
  out->expert_offsets = (int64_t)L.offsets;
  out->gather_idx = (int64_t)L.gather;
  out->slot_pos = (int64_t)L.slotpos;
  out->h = (int64_t)L.h;
  out->h_shared = pb->I_shared > 0 ? (int64_t)L.hs : -1;
  out->h_scales = L.mx_dec ? (int64_t)L.hsc : -1;
  out->h_shared_scales = L.mx_dec && pb->I_shared > 0 ? (int64_t)L.hss : -1;
  return MOE_OK;
}

moe_status moe_router_logits(const moe_problem* pb, const void* x, const void* W_router,
                             const float* router_bias, float* logits, void* workspace,
                             size_t workspace_bytes, void* stream) {
  NvtxRange range("moe_router_logits");
  moe_status s = check_problem(pb);
  if (s != MOE_OK) return s;
  const Layout L = layout_of(*pb);
  if (pb->T == 0) return MOE_OK;
  if (!x || !W_router || !logits) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_router) || !aligned16(logits) ||
      (router_bias && !aligned16(router_bias)))
    return MOE_ERR_INVALID_ARG;
  if ((s = check_ws(workspace, workspace_bytes, L.total)) != MOE_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  const int T = (int)pb->T, H = (int)pb->H, E = (int)pb->E;
  const unsigned long long limit = gemm_problem(*pb).limit_ns;
  if (L.S == 1)
    return cuda_status(launch_router_logits(pb->dtype, x, W_router, router_bias, T, H, E, 1,
                                            logits, status_ptr(workspace), limit, st));
  float* part = at<float>(workspace, L.partials);
  cudaError_t e = launch_router_logits(pb->dtype, x, W_router, router_bias, T, H, E, L.S, part,
                                       status_ptr(workspace), limit, st);
  if (e == cudaSuccess) e = launch_logits_reduce(part, L.S, T, E, router_bias, logits, sm_count(), st);
  return cuda_status(e);
}

moe_status moe_route(const float* logits, int64_t T, int64_t E, int64_t k, int renorm,
                     int32_t* topk_ids, float* topk_w, void* stream) {
  NvtxRange range("moe_route");
  if (T < 0 || E <= 0 || E > 1024 || k <= 0 || k > E || k > 32) return MOE_ERR_INVALID_ARG;
  if (renorm != 0 && renorm != 1) return MOE_ERR_INVALID_ARG;
  if (T * E >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_route(logits, 1, nullptr, (int)T, (int)E, (int)k, renorm, 1, 1,
                                  nullptr, topk_ids, topk_w, (cudaStream_t)stream));
}

moe_status moe_route_grouped(const float* logits, int64_t T, int64_t E, int64_t k, int renorm,
                             int64_t n_group, int64_t topk_group, int32_t* topk_ids,
                             float* topk_w, void* stream) {
  NvtxRange range("moe_route_grouped");
  if (T < 0 || E <= 0 || E > 1024 || k <= 0 || k > E || k > 32) return MOE_ERR_INVALID_ARG;
  if (renorm != 0 && renorm != 1) return MOE_ERR_INVALID_ARG;
  if (!groups_valid(E, k, n_group, topk_group)) return MOE_ERR_INVALID_ARG;
  if (T * E >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_route(logits, 1, nullptr, (int)T, (int)E, (int)k, renorm,
                                  n_group > 1 ? (int)n_group : 1, (int)topk_group, nullptr,
                                  topk_ids, topk_w, (cudaStream_t)stream));
}

moe_status moe_permute(const int32_t* topk_ids, int64_t T, int64_t E, int64_t k,
                       int has_shared, int32_t* expert_offsets, int32_t* gather_idx,
                       int32_t* slot_pos, void* workspace, size_t workspace_bytes,
                       void* stream) {
  NvtxRange range("moe_permute");
  if (T < 0 || E <= 0 || E > 1024 || k <= 0 || k > E || k > 32) return MOE_ERR_INVALID_ARG;
  if (T * (k + 1) >= ((int64_t)1 << 30)) return MOE_ERR_UNSUPPORTED;
  if (!expert_offsets || (T > 0 && (!topk_ids || !gather_idx || !slot_pos)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(expert_offsets) || (T > 0 && (!aligned16(topk_ids) || !aligned16(gather_idx) ||
                                               !aligned16(slot_pos))))
    return MOE_ERR_INVALID_ARG;
  moe_status s = check_ws(workspace, workspace_bytes,
                          align_up(kHeader + permute_scratch_bytes(T, E, k)));
  if (s != MOE_OK) return s;
  return cuda_status(launch_permute(topk_ids, (int)T, (int)E, (int)k, has_shared ? 1 : 0,
                                    expert_offsets, gather_idx, slot_pos,
                                    status_ptr(workspace), at<int32_t>(workspace, kHeader),
                                    (cudaStream_t)stream));
}

moe_status moe_grouped_swiglu_gemm(const moe_problem* pb, const void* x,
                                   const int32_t* expert_offsets, const int32_t* gather_idx,
                                   const int32_t* slot_pos, const void* W_gate, const void* W_up,
                                   const void* Ws_gate, const void* Ws_up, void* h,
                                   void* h_shared, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  NvtxRange range("moe_grouped_swiglu_gemm");
  moe_status s = check_problem(pb);
  if (s != MOE_OK) return s;
  if (pb->T == 0) return MOE_OK;
  const bool has_s = pb->I_shared > 0;
  if (!x || !expert_offsets || !gather_idx || !slot_pos || !W_gate || !W_up || !h)
    return MOE_ERR_INVALID_ARG;
  if (has_s != (Ws_gate != nullptr) || has_s != (Ws_up != nullptr) ||
      has_s != (h_shared != nullptr))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, expert_offsets, gather_idx, slot_pos, W_gate, W_up, h};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (has_s && (!aligned16(Ws_gate) || !aligned16(Ws_up) || !aligned16(h_shared)))
    return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(*pb);
  if ((s = check_ws(workspace, workspace_bytes, L.total)) != MOE_OK) return s;
  if (!tensor_map_encoder_available()) return MOE_ERR_UNSUPPORTED;
  const GemmProblem g = gemm_problem(*pb);
  cudaStream_t st = (cudaStream_t)stream;
  void* xg = nullptr;
  cudaError_t e = cudaSuccess;
  if (gemm_needs_expert_order_copy(g)) {
    xg = at<void>(workspace, L.xg);
    e = launch_gather_rows(x, slot_pos, g.T * g.k, g.k, (size_t)g.H * elem_bytes(g.dtype), xg,
                           status_ptr(workspace), g.num_sms, st);
  }
  if (e == cudaSuccess)
    e = launch_swiglu_gemm(g, x, xg, expert_offsets, gather_idx, W_gate, W_up, Ws_gate, Ws_up, h,
                           h_shared, status_ptr(workspace), st);
  return cuda_status(e);
}

moe_status moe_down_combine(const moe_problem* pb, const void* h, const void* h_shared,
                            const int32_t* expert_offsets, const int32_t* gather_idx,
                            const float* topk_w, const void* W_down, const void* Ws_down,
                            void* y, void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange range("moe_down_combine");
  moe_status s = check_problem(pb);
  if (s != MOE_OK) return s;
  if (pb->T == 0) return MOE_OK;
  const bool has_s = pb->I_shared > 0;
  if (!h || !expert_offsets || !gather_idx || !topk_w || !W_down || !y) return MOE_ERR_INVALID_ARG;
  if (has_s != (Ws_down != nullptr) || has_s != (h_shared != nullptr)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {h, expert_offsets, gather_idx, topk_w, W_down, y};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (has_s && (!aligned16(Ws_down) || !aligned16(h_shared))) return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(*pb);
  if ((s = check_ws(workspace, workspace_bytes, L.total)) != MOE_OK) return s;
  if (!tensor_map_encoder_available()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  const GemmProblem g = gemm_problem(*pb);
  float* Y = at<float>(workspace, L.Y);
  cudaError_t e = launch_down_gemm(g, h, h_shared, expert_offsets, gather_idx, topk_w, W_down,
                                   Ws_down, Y, status_ptr(workspace), st);
  if (e == cudaSuccess)
    e = launch_combine(pb->out_f32 ? MOE_DTYPE_F32 : pb->dtype, Y, g.T, g.H,
                       g.k + (has_s ? 1 : 0), y, g.num_sms, st);
  return cuda_status(e);
}

moe_status moe_forward(const moe_problem* pb, const void* x, const void* W_router,
                       const float* router_bias, const void* W_gate, const void* W_up,
                       const void* W_down, const void* Ws_gate, const void* Ws_up,
                       const void* Ws_down, void* y, void* workspace,
                       size_t workspace_bytes, void* stream) {
  NvtxRange range("moe_forward");
  moe_status s = check_problem(pb);
  if (s != MOE_OK) return s;
  if (pb->T == 0) return MOE_OK;
  const bool has_s = pb->I_shared > 0;
  if (!x || !W_router || !W_gate || !W_up || !W_down || !y) return MOE_ERR_INVALID_ARG;
  if (has_s != (Ws_gate != nullptr) || has_s != (Ws_up != nullptr) ||
      has_s != (Ws_down != nullptr))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, W_router, W_gate, W_up, W_down, y};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (router_bias && !aligned16(router_bias)) return MOE_ERR_INVALID_ARG;
  if (has_s && (!aligned16(Ws_gate) || !aligned16(Ws_up) || !aligned16(Ws_down)))
    return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(*pb);
  if ((s = check_ws(workspace, workspace_bytes, L.total)) != MOE_OK) return s;
  if (!tensor_map_encoder_available()) return MOE_ERR_UNSUPPORTED;

  cudaStream_t st = (cudaStream_t)stream;
  const GemmProblem g = gemm_problem(*pb);
  int* status = status_ptr(workspace);
  float* logits = at<float>(workspace, L.logits);
  float* part = at<float>(workspace, L.partials);
  int32_t* ids = at<int32_t>(workspace, L.ids);
  float* w = at<float>(workspace, L.w);
  int32_t* offs = at<int32_t>(workspace, L.offsets);
  int32_t* gidx = at<int32_t>(workspace, L.gather);
  int32_t* spos = at<int32_t>(workspace, L.slotpos);
  void* h = at<void>(workspace, L.h);
  void* hs = has_s ? at<void>(workspace, L.hs) : nullptr;
  float* Y = at<float>(workspace, L.Y);

  cudaError_t e = cudaMemsetAsync(status, 0, kHeaderClear, st);
  if (e == cudaSuccess) {
    NvtxRange r("router_logits");
    e = launch_router_logits(pb->dtype, x, W_router, router_bias, g.T, g.H, g.E, L.S, part,
                             status, g.limit_ns, st);
  }
  if (e == cudaSuccess) {
    NvtxRange r("route");
    e = launch_route(part, L.S, router_bias, g.T, g.E, g.k, pb->renorm,
                     pb->n_group > 1 ? pb->n_group : 1, pb->topk_group,
                     L.S > 1 ? logits : nullptr, ids, w, st);
  }
  if (e == cudaSuccess) {
    NvtxRange r("permute");
    e = launch_permute(ids, g.T, g.E, g.k, has_s ? 1 : 0, offs, gidx, spos, status,
                       at<int32_t>(workspace, L.pscratch), st);
  }
  void* xg = nullptr;
  if (e == cudaSuccess && gemm_needs_expert_order_copy(g)) {
    NvtxRange r("dispatch_copy");
    xg = at<void>(workspace, L.xg);
    e = launch_gather_rows(x, spos, g.T * g.k, g.k, (size_t)g.H * elem_bytes(g.dtype), xg,
                           status, g.num_sms, st);
  }
  if (e == cudaSuccess) {
    NvtxRange r("gate_up_gemm");
    e = launch_swiglu_gemm(g, x, xg, offs, gidx, W_gate, W_up, Ws_gate, Ws_up, h, hs, status,
                           st);
  }
  if (e == cudaSuccess) {
    NvtxRange r("down_gemm");
    e = launch_down_gemm(g, h, hs, offs, gidx, w, W_down, Ws_down, Y, status, st);
  }
  if (e == cudaSuccess) {
    NvtxRange r("combine");
    e = launch_combine(pb->out_f32 ? MOE_DTYPE_F32 : pb->dtype, Y, g.T, g.H,
                       g.k + (has_s ? 1 : 0), y, g.num_sms, st);
  }
  return cuda_status(e);
}

moe_status moe_forward_single_launch(const moe_problem* pb, const void* x, const void* W_router,
                                     const float* router_bias, const void* W_gate,
                                     const void* W_up, const void* W_down, const void* Ws_gate,
                                     const void* Ws_up, const void* Ws_down, void* y,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange range("moe_forward_single_launch");
  moe_status s = check_problem(pb);
  if (s != MOE_OK) return s;
  if (pb->T == 0) return MOE_OK;
  const bool has_s = pb->I_shared > 0;
  if (!x || !W_router || !W_gate || !W_up || !W_down || !y) return MOE_ERR_INVALID_ARG;
  if (has_s != (Ws_gate != nullptr) || has_s != (Ws_up != nullptr) ||
      has_s != (Ws_down != nullptr))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, W_router, W_gate, W_up, W_down, y};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (router_bias && !aligned16(router_bias)) return MOE_ERR_INVALID_ARG;
  if (has_s && (!aligned16(Ws_gate) || !aligned16(Ws_up) || !aligned16(Ws_down)))
    return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(*pb);
  if ((s = check_ws(workspace, workspace_bytes, L.total)) != MOE_OK) return s;
  if (!tensor_map_encoder_available()) return MOE_ERR_UNSUPPORTED;
  const GemmProblem g = gemm_problem(*pb);
  if (pb->T > 64 || !fused_decode_supported(g)) return MOE_ERR_UNSUPPORTED;

  cudaStream_t st = (cudaStream_t)stream;
  int* status = status_ptr(workspace);
  FusedDecodeIO io;
  io.x = x;
  io.Wr = W_router;
  io.bias = router_bias;
  io.renorm = pb->renorm;
  io.n_group = pb->n_group;
  io.topk_group = pb->topk_group;
  io.out_f32 = pb->out_f32;
  io.Wg = W_gate;
  io.Wu = W_up;
  io.Wd = W_down;
  io.Wsg = Ws_gate;
  io.Wsu = Ws_up;
  io.Wsd = Ws_down;
  io.logits = at<float>(workspace, L.logits);
  io.ids = at<int32_t>(workspace, L.ids);
  io.w = at<float>(workspace, L.w);
  io.offsets = at<int32_t>(workspace, L.offsets);
  io.gather_idx = at<int32_t>(workspace, L.gather);
  io.slot_pos = at<int32_t>(workspace, L.slotpos);
  io.h = at<void>(workspace, L.h);
  io.hs = has_s ? at<void>(workspace, L.hs) : nullptr;
  io.Y = at<float>(workspace, L.Y);
  io.y = y;
  io.status = status;
  io.grid_ctr = status + kGridCounter;
  io.unit_done = at<int>(workspace, L.units);
  io.router_part = at<float>(workspace, L.fpart);
  // The status word and the grid-barrier counter start at zero; the rest is
  // one kernel.
  cudaError_t e = cudaMemsetAsync(status, 0, kHeaderClear, st);
  if (e == cudaSuccess) e = launch_fused_decode(g, io, st);
  return cuda_status(e);
}

moe_status moe_quantize_rows_e4m3(const void* src, int32_t src_dtype, int64_t rows,
                                  int64_t cols, uint8_t* q, float* scale, void* stream) {
  NvtxRange range("moe_quantize_rows_e4m3");
  if (src_dtype != MOE_DTYPE_BF16 && src_dtype != MOE_DTYPE_F32) return MOE_ERR_INVALID_ARG;
  if (rows < 0 || cols <= 0 || cols % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (cols >= ((int64_t)1 << 30)) return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  if (!src || !q || !scale) return MOE_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(q) || !aligned16(scale)) return MOE_ERR_INVALID_ARG;
  return cuda_status(
      launch_quantize_rows(src_dtype, src, rows, cols, q, scale, sm_count(), (cudaStream_t)stream));
}

moe_status moe_forward_fp8(const moe_problem* pb, const void* x, const void* W_router,
                           const float* router_bias, const uint8_t* Wq_gate, const float* s_gate,
                           const uint8_t* Wq_up, const float* s_up, const uint8_t* Wq_down,
                           const float* s_down, const uint8_t* Wsq_gate, const float* ss_gate,
                           const uint8_t* Wsq_up, const float* ss_up, const uint8_t* Wsq_down,
                           const float* ss_down, void* y, void* workspace,
                           size_t workspace_bytes, void* stream) {
  NvtxRange range("moe_forward_fp8");
  if (!pb || pb->dtype != MOE_DTYPE_E4M3) return MOE_ERR_INVALID_ARG;
  moe_status s = check_problem(pb, true);
  if (s != MOE_OK) return s;
  if (pb->T == 0) return MOE_OK;
  const bool has_s = pb->I_shared > 0;
  const void* ptrs[] = {x, W_router, Wq_gate, s_gate, Wq_up, s_up, Wq_down, s_down, y};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (router_bias && !aligned16(router_bias)) return MOE_ERR_INVALID_ARG;
  const void* sptrs[] = {Wsq_gate, ss_gate, Wsq_up, ss_up, Wsq_down, ss_down};
  for (const void* q : sptrs) {
    if (has_s != (q != nullptr)) return MOE_ERR_INVALID_ARG;
    if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
  }
  const Layout L = layout_of(*pb);
  if ((s = check_ws(workspace, workspace_bytes, L.total)) != MOE_OK) return s;
  if (!tensor_map_encoder_available()) return MOE_ERR_UNSUPPORTED;

  cudaStream_t st = (cudaStream_t)stream;
  const GemmProblem g = gemm_problem(*pb);  // dtype E4M3: the expert GEMMs
  int* status = status_ptr(workspace);
  float* logits = at<float>(workspace, L.logits);
  float* part = at<float>(workspace, L.partials);
  int32_t* ids = at<int32_t>(workspace, L.ids);
  float* w = at<float>(workspace, L.w);
  int32_t* offs = at<int32_t>(workspace, L.offsets);
  int32_t* gidx = at<int32_t>(workspace, L.gather);
  int32_t* spos = at<int32_t>(workspace, L.slotpos);
  uint8_t* xq = at<uint8_t>(workspace, L.xq);
  float* sx = at<float>(workspace, L.sx);
  void* h = at<void>(workspace, L.h);
  void* hs = has_s ? at<void>(workspace, L.hs) : nullptr;
  uint8_t* hq = at<uint8_t>(workspace, L.hq);
  float* sh = at<float>(workspace, L.sh);
  uint8_t* hsq = has_s ? at<uint8_t>(workspace, L.hsq) : nullptr;
  float* shs = has_s ? at<float>(workspace, L.shs) : nullptr;
  float* Y = at<float>(workspace, L.Y);

  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), st);
  // Router, routing and permutation exactly as the bf16 layer.
  if (e == cudaSuccess)
    e = launch_router_logits(MOE_DTYPE_BF16, x, W_router, router_bias, g.T, g.H, g.E, L.S, part,
                             status, g.limit_ns, st);
  if (e == cudaSuccess)
    e = launch_route(part, L.S, router_bias, g.T, g.E, g.k, pb->renorm,
                     pb->n_group > 1 ? pb->n_group : 1, pb->topk_group,
                     L.S > 1 ? logits : nullptr, ids, w, st);
  if (e == cudaSuccess)
    e = launch_permute(ids, g.T, g.E, g.k, has_s ? 1 : 0, offs, gidx, spos, status,
                       at<int32_t>(workspace, L.pscratch), st);
  // Token rows to E4M3 (one scale per token), then the expert-ordered copy of
  // the codes when the tiled kernel runs.
  if (e == cudaSuccess)
    e = launch_quantize_rows(MOE_DTYPE_BF16, x, g.T, g.H, xq, sx, g.num_sms, st);
  void* xg = nullptr;
  if (e == cudaSuccess && gemm_needs_expert_order_copy(g)) {
    xg = at<void>(workspace, L.xg);
    e = launch_gather_rows(xq, spos, g.T * g.k, g.k, (size_t)g.H, xg, status, g.num_sms, st);
  }
  GemmScales sg = {{s_gate, s_up, ss_gate, ss_up}, {sx, sx}};
  if (e == cudaSuccess)
    e = launch_swiglu_gemm(g, xq, xg, offs, gidx, Wq_gate, Wq_up, Wsq_gate, Wsq_up, h, hs, status,
                           st, &sg);
  // h rows (bf16) to E4M3, one scale per row, for the down projection.
  if (e == cudaSuccess)
    e = launch_quantize_rows(MOE_DTYPE_BF16, h, (int64_t)g.T * g.k, g.I, hq, sh, g.num_sms, st);
  if (e == cudaSuccess && has_s)
    e = launch_quantize_rows(MOE_DTYPE_BF16, hs, g.T, g.Is, hsq, shs, g.num_sms, st);
  GemmScales sd = {{s_down, nullptr, ss_down, nullptr}, {sh, shs}};
  if (e == cudaSuccess)
    e = launch_down_gemm(g, hq, hsq, offs, gidx, w, Wq_down, Wsq_down, Y, status, st, &sd);
  if (e == cudaSuccess)
    e = launch_combine(pb->out_f32 ? MOE_DTYPE_F32 : MOE_DTYPE_BF16, Y, g.T, g.H,
                       g.k + (has_s ? 1 : 0), y, g.num_sms, st);
  return cuda_status(e);
}

int64_t moe_mx_scale_cols(int64_t cols) { return cols < 0 ? 0 : 16 * ((cols / 32 + 15) / 16); }

moe_status moe_quantize_mx(const void* src, int32_t src_dtype, int64_t rows, int64_t cols,
                           uint8_t* q, uint8_t* scales, void* stream) {
  NvtxRange range("moe_quantize_mx");
  if (src_dtype != MOE_DTYPE_BF16 && src_dtype != MOE_DTYPE_F32) return MOE_ERR_INVALID_ARG;
  if (rows < 0 || cols <= 0 || cols % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (cols >= ((int64_t)1 << 30) || rows * moe_mx_scale_cols(cols) >= ((int64_t)1 << 40))
    return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  if (!src || !q || !scales) return MOE_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(q) || !aligned16(scales)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_mx(src_dtype, src, rows, cols, q, scales, sm_count(),
                                        (cudaStream_t)stream));
}

moe_status moe_forward_mx(const moe_problem* pb, const void* x, const void* W_router,
                          const float* router_bias, const uint8_t* Wq_gate, const uint8_t* s_gate,
                          const uint8_t* Wq_up, const uint8_t* s_up, const uint8_t* Wq_down,
                          const uint8_t* s_down, const uint8_t* Wsq_gate, const uint8_t* ss_gate,
                          const uint8_t* Wsq_up, const uint8_t* ss_up, const uint8_t* Wsq_down,
                          const uint8_t* ss_down, void* y, void* workspace,
                          size_t workspace_bytes, void* stream) {
  NvtxRange range("moe_forward_mx");
  if (!pb || pb->dtype != MOE_DTYPE_MXFP8) return MOE_ERR_INVALID_ARG;
  moe_status s = check_problem(pb, true);
  if (s != MOE_OK) return s;
  if (pb->T == 0) return MOE_OK;
  const bool has_s = pb->I_shared > 0;
  const void* ptrs[] = {x, W_router, Wq_gate, s_gate, Wq_up, s_up, Wq_down, s_down, y};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (router_bias && !aligned16(router_bias)) return MOE_ERR_INVALID_ARG;
  const void* sptrs[] = {Wsq_gate, ss_gate, Wsq_up, ss_up, Wsq_down, ss_down};
  for (const void* p : sptrs) {
    if (has_s != (p != nullptr)) return MOE_ERR_INVALID_ARG;
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  }
  const Layout L = layout_of(*pb);
  if ((s = check_ws(workspace, workspace_bytes, L.total)) != MOE_OK) return s;
  if (!tensor_map_encoder_available()) return MOE_ERR_UNSUPPORTED;
  const GemmProblem g = gemm_problem(*pb);
  if (!mx_problem_fits(g)) return MOE_ERR_UNSUPPORTED;

  cudaStream_t st = (cudaStream_t)stream;
  int* status = status_ptr(workspace);
  float* logits = at<float>(workspace, L.logits);
  float* part = at<float>(workspace, L.partials);
  int32_t* ids = at<int32_t>(workspace, L.ids);
  float* w = at<float>(workspace, L.w);
  int32_t* offs = at<int32_t>(workspace, L.offsets);
  int32_t* gidx = at<int32_t>(workspace, L.gather);
  int32_t* spos = at<int32_t>(workspace, L.slotpos);
  void* xm = L.xm ? at<void>(workspace, L.xm) : nullptr;
  void* xg = at<void>(workspace, L.xg);
  void* h = at<void>(workspace, L.h);
  void* hs = has_s ? at<void>(workspace, L.hs) : nullptr;
  float* Y = at<float>(workspace, L.Y);
  const MxWeights mw = {Wq_gate, s_gate, Wq_up, s_up, Wq_down, s_down,
                        Wsq_gate, ss_gate, Wsq_up, ss_up, Wsq_down, ss_down};

  cudaError_t e = cudaMemsetAsync(status, 0, kHeaderClear, st);
  // Router, routing and permutation exactly as the bf16 layer (on x itself).
  if (e == cudaSuccess) {
    NvtxRange r("router_logits");
    e = launch_router_logits(MOE_DTYPE_BF16, x, W_router, router_bias, g.T, g.H, g.E, L.S, part,
                             status, g.limit_ns, st);
  }
  if (e == cudaSuccess) {
    NvtxRange r("route");
    e = launch_route(part, L.S, router_bias, g.T, g.E, g.k, pb->renorm,
                     pb->n_group > 1 ? pb->n_group : 1, pb->topk_group,
                     L.S > 1 ? logits : nullptr, ids, w, st);
  }
  if (e == cudaSuccess) {
    NvtxRange r("permute");
    e = launch_permute(ids, g.T, g.E, g.k, has_s ? 1 : 0, offs, gidx, spos, status,
                       at<int32_t>(workspace, L.pscratch), st);
  }
  if (L.mx_dec) {
    // Decode-sized batches: token rows to MXFP8 codes and scale rows, written
    // in expert order (and token order for a shared expert), then the E4M3-MMA
    // GEMMs (h as codes and scales).
    uint8_t* xq = at<uint8_t>(workspace, L.xq);
    uint8_t* xs = at<uint8_t>(workspace, L.xs);
    uint8_t* xgq = at<uint8_t>(workspace, L.xg);
    uint8_t* xgs = at<uint8_t>(workspace, L.xgs);
    const MxDecTokens xt = {xgq, xgs, xq, xs};
    const MxDecOut ho = {at<uint8_t>(workspace, L.h), at<uint8_t>(workspace, L.hsc),
                         has_s ? at<uint8_t>(workspace, L.hs) : nullptr,
                         has_s ? at<uint8_t>(workspace, L.hss) : nullptr};
    const MxDecTokens ht = {ho.routed, ho.routed_scales, ho.shared, ho.shared_scales};
    if (e == cudaSuccess) {
      NvtxRange r("quantize_dispatch_x");
      e = launch_quantize_dispatch_mx(x, spos, g.T, g.k, g.H, xgq, xgs, has_s ? xq : nullptr,
                                      has_s ? xs : nullptr, status, g.num_sms, st);
    }
    if (e == cudaSuccess) {
      NvtxRange r("gate_up_gemm");
      e = launch_mx_dec_swiglu_gemm(g, mw, xt, offs, gidx, ho, status, st);
    }
    if (e == cudaSuccess) {
      NvtxRange r("down_gemm");
      e = launch_mx_dec_down_gemm(g, mw, ht, offs, gidx, w, Y, status, st);
    }
  } else {
    // Token rows to their MXFP8 values (bf16), then their expert-ordered copy.
    if (e == cudaSuccess) {
      NvtxRange r("quantize_x");
      e = launch_qdq_mx(x, g.T, g.H, xm, g.num_sms, st);
    }
    if (e == cudaSuccess) {
      NvtxRange r("dispatch_copy");
      e = launch_gather_rows(xm, spos, g.T * g.k, g.k, (size_t)g.H * 2, xg, status, g.num_sms,
                             st);
    }
    if (e == cudaSuccess) {
      NvtxRange r("gate_up_gemm");
      e = launch_mx_swiglu_gemm(g, mw, xm, xg, offs, gidx, h, hs, status, st);
    }
    if (e == cudaSuccess) {
      NvtxRange r("down_gemm");
      e = launch_mx_down_gemm(g, mw, h, hs, offs, gidx, w, Y, status, st);
    }
  }
  if (e == cudaSuccess) {
    NvtxRange r("combine");
    e = launch_combine(pb->out_f32 ? MOE_DTYPE_F32 : MOE_DTYPE_BF16, Y, g.T, g.H,
                       g.k + (has_s ? 1 : 0), y, g.num_sms, st);
  }
  return cuda_status(e);
}

moe_status moe_get_device_status(const void* workspace, void* stream, moe_status* out) {
  if (!workspace || !out) return MOE_ERR_INVALID_ARG;
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  *out = (moe_status)v;
  return MOE_OK;
}

moe_status moe_reset_device_status(void* workspace, void* stream) {
  if (!workspace) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(workspace, 0, sizeof(int), (cudaStream_t)stream));
}

}  // extern "C"
