// Single-launch decode path: the whole layer (router logits, top-k routing,
// permutation, gate/up GEMM with SwiGLU, down GEMM, combine) in one persistent
// kernel for decode-sized batches (the 32-token decode tiles).
//
// "Lower latency and higher throughput with multi-node DeepSeek deployment"
// (its CUDA-Graph paragraph) describes persistent kernels that read the
// per-expert counts on the device so that a decode step replays without host
// work, and the "CuTeDSL at Perplexity" decode dispatch runs the small-batch
// routing inside the same kernel as the data movement. Here one cooperative
// launch with one CTA per SM runs:
//  1. the router logits, split over all CTAs: a CTA takes 8 experts and one
//     slice of H for every token and writes fp32 partial sums (a fixed order
//     within the slice); meanwhile every CTA asks L2 for the weight rows of its
//     likely first gate/up unit;
//  2. a grid barrier; one warp per token adds its slices in ascending order
//     (plus the bias) and routes the token (the route kernel's warp routine);
//     a grid barrier; every CTA computes the stable permutation itself into
//     its own shared memory (CTA 0 also stores it for the caller);
//  3. the gate/up GEMM pass (the decode kernel's, same schedule); each unit
//     counts itself done for its expert once its h rows are stored;
//  4. the down GEMM pass; before loading an expert's h rows, a unit waits
//     until all of that expert's gate/up units are done, so CTAs that finish
//     their gate/up units early start on the down GEMM while others finish
//     theirs (no kernel boundary between the two GEMMs);
//  5. a third grid barrier, then the rank-order combine.
// Every wait is bounded (wait_limit_us) and gives up once the status word is
// set; the cooperative launch guarantees that all CTAs are resident together,
// which the cross-CTA waits need.
#include <cmath>
#include <mutex>

#include "combine.cuh"
#include "common.cuh"
#include "grouped_gemm.cuh"
#include "kernels.h"
#include "permute_block.cuh"
#include "route_warp.cuh"

namespace moe {

namespace {

constexpr int FD_BN = 32;      // the decode GEMMs' token tile
constexpr int FD_STAGES = 9;   // and their ring depth
constexpr int FD_WARPS = 6;    // producer, MMA issuer, four epilogue warps
constexpr int FD_THREADS = FD_WARPS * 32;

template <typename TIn>
using FdGated = GemmCfg<TIn, true, FD_BN, FD_STAGES, kGather4, 1>;
template <typename TIn>
using FdDown = GemmCfg<TIn, false, FD_BN, FD_STAGES, kTiled, 1>;
static_assert(FdGated<__nv_bfloat16>::THREADS == FD_THREADS &&
                  FdDown<__nv_bfloat16>::THREADS == FD_THREADS &&
                  FdGated<float>::THREADS == FD_THREADS && FdDown<float>::THREADS == FD_THREADS,
              "both passes run on the same 6 warps");

struct FusedDecodeArgs {
  GroupedGemmArgs gated, down;  // as launch_swiglu_gemm / launch_down_gemm build them
  const void* x;
  const void* Wr;
  const float* bias;
  float* logits;                // [T][E]
  int32_t* ids;                 // [T][k]
  float* w;                     // [T][k]
  int32_t* offsets;             // [E+2]   (copies of the permutation, for the caller)
  int32_t* gather_idx;          // [T*k]
  int32_t* slot_pos;            // [T*k]
  const float* Y;               // slot rows [T][KP][H]
  void* y;                      // [T][H]
  float* part;                  // router partial sums [S][T][E]
  int* status;
  int* grid_ctr;                // zero at launch
  int* unit_done;               // [E+1], zeroed here before the first barrier
  unsigned long long limit_ns;
  int T, H, E, k, KP, renorm, n_group, topk_group, has_shared, out_f32;
  int S, Ls;                    // router slices of H and their length
  int perm_off;                 // byte offset of the permutation copies in shared memory
};

constexpr int FD_RB = 8;        // experts per router work item

// All CTAs of the grid. The arrivals are counted on *ctr; `target` is the
// count after this barrier (G for the first, 2G for the second). Bounded.
__device__ __forceinline__ bool grid_sync(int* ctr, int target, int* status, uint64_t limit,
                                          volatile int* flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    red_release_gpu_add(ctr, 1);
    const bool ok = wait_count_at_least(ctr, target, status, limit);
    __threadfence();
    *flag = ok ? 1 : 0;
  }
  __syncthreads();
  return *flag != 0;
}

template <typename TIn>
__device__ __forceinline__ void load8_f32(const TIn* p, float (&v)[8]);
template <>
__device__ __forceinline__ void load8_f32<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(b[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
template <>
__device__ __forceinline__ void load8_f32<float>(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// 16-byte asynchronous copy global -> shared (no register round trip), and the
// wait for all of this thread's copies.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Step 1, one work item: partial logits of experts e0..e0+7 over the H slice
// [h0, h0 + len) for every token, into part[s][t][e]. The 8 weight rows and
// every token's x slice are copied into shared memory first (asynchronous
// 16-byte copies, all in flight together), each row padded by 16 bytes so
// that rows fall on different banks. Lane (q, j) of warp w, q < 4, j < 8, then
// computes the dot product of token w * 4 + q + 24 i with expert e0 + j over
// the whole slice: four running sums over the slice's 16-element chunks
// (elements 4m..4m+3 of a chunk to sum m), added as (s0 + s1) + (s2 + s3) at
// the end. One lane per dot product: no cross-lane reduction.
template <typename TIn>
__device__ void router_item(const FusedDecodeArgs& a, int e0, int s, uint8_t* scratch) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h0 = s * a.Ls, len = min(a.Ls, a.H - h0);
  const int ne = min(FD_RB, a.E - e0);
  const TIn* Wr = static_cast<const TIn*>(a.Wr);
  const TIn* x = static_cast<const TIn*>(a.x);
  constexpr int VX = 16 / (int)sizeof(TIn);  // elements per 16 bytes
  const int ld = len + VX;                    // padded row stride (elements)
  TIn* ws = reinterpret_cast<TIn*>(scratch);
  TIn* xs = ws + FD_RB * ld;
  const int nw = ne * len, nx = a.T * len;
  for (int i = threadIdx.x * VX; i < nw + nx; i += FD_THREADS * VX) {
    if (i < nw) {
      const int j = i / len, c = i - j * len;
      cp_async16(ws + j * ld + c, Wr + (size_t)(e0 + j) * a.H + h0 + c);
    } else {
      const int t = (i - nw) / len, c = (i - nw) - t * len;
      cp_async16(xs + (size_t)t * ld + c, x + (size_t)t * a.H + h0 + c);
    }
  }
  cp_async_wait_all();
  __syncthreads();
  const int q = lane >> 3, j = lane & 7;
  const TIn* wrow = ws + min(j, ne - 1) * ld;
  for (int t0 = warp * 4; t0 < a.T; t0 += FD_WARPS * 4) {
    const int t = t0 + q;
    const TIn* xrow = xs + (size_t)min(t, a.T - 1) * ld;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    for (int c = 0; c < len; c += 16) {
      float xa[8], xb[8], wa[8], wb[8];
      load8_f32<TIn>(xrow + c, xa);
      load8_f32<TIn>(xrow + c + 8, xb);
      load8_f32<TIn>(wrow + c, wa);
      load8_f32<TIn>(wrow + c + 8, wb);
      s0 = fmaf(xa[0], wa[0], s0);
      s0 = fmaf(xa[1], wa[1], s0);
      s0 = fmaf(xa[2], wa[2], s0);
      s0 = fmaf(xa[3], wa[3], s0);
      s1 = fmaf(xa[4], wa[4], s1);
      s1 = fmaf(xa[5], wa[5], s1);
      s1 = fmaf(xa[6], wa[6], s1);
      s1 = fmaf(xa[7], wa[7], s1);
      s2 = fmaf(xb[0], wb[0], s2);
      s2 = fmaf(xb[1], wb[1], s2);
      s2 = fmaf(xb[2], wb[2], s2);
      s2 = fmaf(xb[3], wb[3], s2);
      s3 = fmaf(xb[4], wb[4], s3);
      s3 = fmaf(xb[5], wb[5], s3);
      s3 = fmaf(xb[6], wb[6], s3);
      s3 = fmaf(xb[7], wb[7], s3);
    }
    if (t < a.T && j < ne) a.part[((size_t)s * a.T + t) * a.E + e0 + j] = (s0 + s1) + (s2 + s3);
  }
  __syncthreads();  // the scratch is rewritten by the next item
}

// Step 2 for token t by one warp: logits = the slices' partial sums added in
// ascending slice order, plus the bias (written out), then top-k and weights.
template <int NV>
__device__ __forceinline__ void route_token_warp(const FusedDecodeArgs& a, int t) {
  const int lane = threadIdx.x & 31;
  float v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    float acc = -INFINITY;
    if (e < a.E) {
      // All slices' loads first (one round trip), then the sum in slice order.
      float q[8];
#pragma unroll
      for (int s = 0; s < 8; ++s)
        q[s] = s < a.S ? __ldcg(a.part + ((size_t)s * a.T + t) * a.E + e) : 0.f;
      acc = q[0];
#pragma unroll
      for (int s = 1; s < 8; ++s)
        if (s < a.S) acc += q[s];
      if (a.bias) acc += a.bias[e];
      if (a.logits) a.logits[(size_t)t * a.E + e] = acc;
    }
    v[i] = acc;
  }
  route_warp<NV>(v, a.E, a.k, a.renorm, a.n_group, a.topk_group, a.ids + (size_t)t * a.k,
                 a.w + (size_t)t * a.k);
}

__device__ __forceinline__ void route_token_any(const FusedDecodeArgs& a, int t) {
  const int nv = (a.E + 31) / 32;
  if (nv <= 1) route_token_warp<1>(a, t);
  else if (nv <= 2) route_token_warp<2>(a, t);
  else if (nv <= 4) route_token_warp<4>(a, t);
  else if (nv <= 8) route_token_warp<8>(a, t);
  else if (nv <= 16) route_token_warp<16>(a, t);
  else route_token_warp<32>(a, t);
}

template <typename TIn>
__global__ void __launch_bounds__(FD_THREADS, 1)
    fused_decode_kernel(const __grid_constant__ FusedDecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // Scratch for steps 1-2 at the start of the GEMM passes' region (their
  // stages), the permutation copies past it.
  uint8_t* scratch = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int32_t* offs_s = reinterpret_cast<int32_t*>(smem_raw + a.perm_off);
  int32_t* gidx_s = offs_s + ((a.E + 2 + 3) & ~3);
  int32_t* spos_s = gidx_s + a.T * a.k;
  volatile int* flag = reinterpret_cast<volatile int*>(spos_s + a.T * a.k);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;

  // 1. Router partial sums, and the per-expert unit counts start at zero.
  if (blockIdx.x == 0)
    for (int g = threadIdx.x; g <= a.E; g += FD_THREADS) a.unit_done[g] = 0;
  const int eb = (a.E + FD_RB - 1) / FD_RB;
  for (int item = blockIdx.x; item < eb * a.S; item += G)
    router_item<TIn>(a, (item % eb) * FD_RB, item / eb, scratch);
  // HBM is otherwise idle until the gate/up GEMM starts: ask L2 for this CTA's
  // likely first gate/up weight rows (as the chained gate/up GEMM does before
  // waiting), once this CTA's router reads are done, so that they do not queue
  // behind 150 MB of prefetch.
  if (warp == 0) prefetch_first_unit<TIn, true, FdGated<TIn>::WM>(a.gated, blockIdx.x, lane);
  bool ok = grid_sync(a.grid_ctr, G, a.status, a.limit_ns, flag);

  // 2. Routing, one warp per token; then the permutation, by every CTA into
  // its own shared memory.
  if (ok) {
    const int t = blockIdx.x * FD_WARPS + warp;
    if (t < a.T) route_token_any(a, t);
  }
  ok = ok && grid_sync(a.grid_ctr, 2 * G, a.status, a.limit_ns, flag);
  if (ok) {
    permute_block<FD_WARPS, true>(a.ids, a.T, a.E, a.k, a.has_shared, offs_s, gidx_s, spos_s,
                                  a.status, reinterpret_cast<int32_t*>(scratch));
    __syncthreads();
    if (blockIdx.x == 0) {
      for (int i = threadIdx.x; i < a.E + 2; i += FD_THREADS) a.offsets[i] = offs_s[i];
      for (int i = threadIdx.x; i < a.T * a.k; i += FD_THREADS) {
        a.gather_idx[i] = gidx_s[i];
        a.slot_pos[i] = spos_s[i];
      }
    }
    // One decision for the whole CTA (every thread then takes the same
    // branches around the passes' block barriers).
    if (threadIdx.x == 0) *flag = read_status(a.status) == MOE_OK ? 1 : 0;
    __syncthreads();
    ok = *flag != 0;
  }

  // 3-4. The two GEMM passes in the same shared memory.
  if (ok)
    grouped_gemm_pass<TIn, true, FD_BN, FD_STAGES, kGather4, 1, true>(
        a.gated, smem_raw, blockIdx.x, G, false, offs_s, gidx_s, /*last_alloc=*/false);
  if (ok)
    grouped_gemm_pass<TIn, false, FD_BN, FD_STAGES, kTiled, 1, true>(
        a.down, smem_raw, blockIdx.x, G, false, offs_s, gidx_s);

  // 5. Every slot row is stored: combine.
  ok = ok && grid_sync(a.grid_ctr, 3 * G, a.status, a.limit_ns, flag);
  if (ok) {
    const size_t i0 = blockIdx.x * (size_t)FD_THREADS + threadIdx.x;
    const size_t step = (size_t)G * FD_THREADS;
    if (a.out_f32)
      combine_range<float>(a.Y, a.T, a.H, a.KP, static_cast<float*>(a.y), i0, step);
    else if constexpr (sizeof(TIn) == 2)
      combine_range<__nv_bfloat16>(a.Y, a.T, a.H, a.KP, static_cast<__nv_bfloat16*>(a.y), i0,
                                   step);
    else
      combine_range<float>(a.Y, a.T, a.H, a.KP, static_cast<float*>(a.y), i0, step);
  }
}

// Shared memory of the kernel: the larger GEMM pass, then the permutation
// copies and the barrier flag.
template <typename TIn>
size_t fused_smem_bytes(int T, int E, int k, size_t* perm_off) {
  size_t pass = FdGated<TIn>::smem_bytes(E);
  if (FdDown<TIn>::smem_bytes(E) > pass) pass = FdDown<TIn>::smem_bytes(E);
  pass = (pass + 15) / 16 * 16;
  *perm_off = pass;
  return pass + ((size_t)((E + 2 + 3) & ~3) + 2 * (size_t)T * k + 4) * 4;
}

// Router split of H: slices of at most 512 unless that would take more than 8
// slices, each a multiple of 64 long (so 16-element chunks tile a slice);
// (E / 8) x S work items are dealt to the CTAs, and an item stages its slice
// of every token in shared memory.
void router_plan(int H, int E, int G, int* S, int* Ls) {
  (void)E;
  (void)G;
  int want = (H + 511) / 512;
  want = want < 1 ? 1 : (want > 8 ? 8 : want);
  int len = (H + want - 1) / want;
  len = (len + 63) / 64 * 64;
  *Ls = len;
  *S = (H + len - 1) / len;
}

// Steps 1-2 keep their scratch inside the passes' stage ring.
template <typename TIn>
bool fused_scratch_fits(int T, int H, int E, int G) {
  const size_t ring = (size_t)FD_STAGES * FdGated<TIn>::STAGE_BYTES;
  int S = 1, Ls = H;
  router_plan(H, E, G, &S, &Ls);
  const size_t route = ((size_t)FD_RB + T) * (Ls + 16 / sizeof(TIn)) * sizeof(TIn);
  const size_t perm = ((size_t)FD_WARPS * E + E + FD_WARPS) * 4;
  return route <= ring && perm <= ring;
}

// Per-device facts the eligibility test needs, looked up once: the opt-in
// shared-memory limit, cooperative-launch support, the kernels' shared memory
// attribute raised to that limit, and whether a CTA using all of it is
// resident (then every smaller one is too).
struct FusedDeviceInfo {
  bool ready = false;
  int optin = 0;
  int coop = 0;
  int resident = 0;
  cudaError_t err = cudaSuccess;
};
std::mutex g_fd_mu;
FusedDeviceInfo g_fd_info[64];

cudaError_t fused_device_info(FusedDeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_fd_mu);
  FusedDeviceInfo& d = g_fd_info[dev];
  if (!d.ready) {
    d.err = cudaDeviceGetAttribute(&d.optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (d.err == cudaSuccess)
      d.err = cudaDeviceGetAttribute(&d.coop, cudaDevAttrCooperativeLaunch, dev);
    if (d.err == cudaSuccess)
      d.err = cudaFuncSetAttribute(fused_decode_kernel<__nv_bfloat16>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, d.optin);
    if (d.err == cudaSuccess)
      d.err = cudaFuncSetAttribute(fused_decode_kernel<float>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, d.optin);
    int bf = 0, f32 = 0;
    if (d.err == cudaSuccess)
      d.err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &bf, fused_decode_kernel<__nv_bfloat16>, FD_THREADS, (size_t)d.optin);
    if (d.err == cudaSuccess)
      d.err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&f32, fused_decode_kernel<float>,
                                                            FD_THREADS, (size_t)d.optin);
    d.resident = (bf >= 1 && f32 >= 1) ? 1 : 0;
    d.ready = true;
  }
  *out = d;
  return d.err;
}

// The kernel's shared memory for this problem, if the device can run it with
// one CTA per SM (its shared memory allows no second CTA); else an error.
template <typename TIn>
cudaError_t fused_check(const GemmProblem& p, size_t* smem, size_t* perm_off, int* grid) {
  if (!fused_scratch_fits<TIn>(p.T, p.H, p.E, p.num_sms)) return cudaErrorInvalidValue;
  *smem = fused_smem_bytes<TIn>(p.T, p.E, p.k, perm_off);
  FusedDeviceInfo info;
  const cudaError_t e = fused_device_info(&info);
  if (e != cudaSuccess) return e;
  if (!info.coop || !info.resident || *smem > (size_t)info.optin) return cudaErrorInvalidValue;
  *grid = p.num_sms;
  return cudaSuccess;
}

template <typename TIn>
cudaError_t launch_fused(const GemmProblem& p, const FusedDecodeIO& io, cudaStream_t st) {
  size_t smem = 0, perm_off = 0;
  int grid = 0;
  cudaError_t e = fused_check<TIn>(p, &smem, &perm_off, &grid);
  if (e != cudaSuccess) return e;
  if (grid * FD_WARPS < p.T) return cudaErrorInvalidValue;  // one warp per token routes it
  FusedDecodeArgs a;
  memset(&a, 0, sizeof(a));
  // The permutation is read from each CTA's shared-memory copy; the argument
  // pointers below are placeholders the passes do not use.
  if (!prepare_swiglu_gemm(a.gated, p, io.x, nullptr, io.offsets, io.gather_idx, io.Wg, io.Wu,
                           io.Wsg, io.Wsu, io.h, io.hs, io.status, nullptr) ||
      !prepare_down_gemm(a.down, p, io.h, io.hs, io.offsets, io.gather_idx, io.w, io.Wd, io.Wsd,
                         io.Y, io.status, nullptr))
    return cudaErrorInvalidValue;
  a.gated.unit_done = io.unit_done;
  a.down.unit_wait = io.unit_done;
  a.down.wait_block = FdGated<TIn>::WM;
  a.x = io.x;
  a.Wr = io.Wr;
  a.bias = io.bias;
  a.logits = io.logits;
  a.ids = io.ids;
  a.w = io.w;
  a.offsets = io.offsets;
  a.gather_idx = io.gather_idx;
  a.slot_pos = io.slot_pos;
  a.Y = io.Y;
  a.y = io.y;
  a.status = io.status;
  a.grid_ctr = io.grid_ctr;
  a.unit_done = io.unit_done;
  a.limit_ns = p.limit_ns;
  a.T = p.T;
  a.H = p.H;
  a.E = p.E;
  a.k = p.k;
  a.KP = p.k + (p.Is > 0 ? 1 : 0);
  a.renorm = io.renorm;
  a.n_group = io.n_group > 1 ? io.n_group : 1;
  a.topk_group = io.topk_group;
  a.has_shared = p.Is > 0 ? 1 : 0;
  a.out_f32 = io.out_f32;
  a.perm_off = (int)perm_off;
  router_plan(p.H, p.E, grid, &a.S, &a.Ls);
  a.part = io.router_part;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(FD_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, fused_decode_kernel<TIn>, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool fused_decode_supported(const GemmProblem& p) {
  if (p.T < 1 || !gemm_uses_decode_tiles(p) || p.T > p.num_sms * FD_WARPS) return false;
  if (p.dtype != MOE_DTYPE_BF16 && p.dtype != MOE_DTYPE_F32) return false;
  size_t smem = 0, perm_off = 0;
  int grid = 0;
  const cudaError_t e = p.dtype == MOE_DTYPE_BF16
                            ? fused_check<__nv_bfloat16>(p, &smem, &perm_off, &grid)
                            : fused_check<float>(p, &smem, &perm_off, &grid);
  return e == cudaSuccess;
}

cudaError_t launch_fused_decode(const GemmProblem& p, const FusedDecodeIO& io, cudaStream_t st) {
  if (p.dtype == MOE_DTYPE_BF16) return launch_fused<__nv_bfloat16>(p, io, st);
  if (p.dtype == MOE_DTYPE_F32) return launch_fused<float>(p, io, st);
  return cudaErrorInvalidValue;
}

}  // namespace moe
