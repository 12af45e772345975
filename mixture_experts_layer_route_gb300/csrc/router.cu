// Router: logits (step a1) and top-k routing with gate weights (step a2).
//
// Logits: logits[t][e] = sum_h x[t][h] * Wr[e][h] (+ b[e]) with fp32
// accumulation ("Gate" at the end of stage 2 of the five-stage MoE layer in
// "Lower latency and higher throughput with multi-node DeepSeek deployment").
// bf16 layers compute it on the tensor cores (tcgen05, bf16 products are exact
// in the fp32 accumulator); fp32 layers on the CUDA cores, since tf32 operands
// would round x and Wr. When the tile grid alone cannot fill the GPU (decode:
// T = 64), H is split into S slices whose partial sums are added later in
// ascending slice order, so results do not depend on scheduling.
//
// Route: one warp per token keeps the token's E logits in registers, takes the
// k largest one at a time (lowest expert index among equal values), then the
// softmax gate weights over the chosen k (renorm) or over all E ("MoE Router"
// section of the same page: top-k indices and scores per token).
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "route_warp.cuh"

namespace moe {

namespace {

constexpr int RT_BM = 64;   // tokens per tile
constexpr int RT_BN = 64;   // experts per tile
constexpr int RT_BK = 32;   // K per smem stage
constexpr int RT_PAD = 4;   // keeps float4 alignment, spreads banks

template <typename TIn>
__device__ __forceinline__ void load_vec_f32(const TIn* p, float* out);

template <>
__device__ __forceinline__ void load_vec_f32<__nv_bfloat16>(const __nv_bfloat16* p, float* out) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(b[i]);
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}

template <>
__device__ __forceinline__ void load_vec_f32<float>(const float* p, float* out) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  out[0] = v.x;
  out[1] = v.y;
  out[2] = v.z;
  out[3] = v.w;
}

// Two fp32 lanes in one 64-bit register; fma.rn.f32x2 performs two IEEE fp32
// FMAs (the same rounding as fmaf) with one instruction.
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ void fma2(unsigned long long& d, unsigned long long a,
                                     unsigned long long b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

// grid (ceil(E/64), ceil(T/64), S); block 256. out: [S][T][E].
// Each thread owns 4 tokens x 4 experts; both operands are staged in shared
// memory as fp32, K-major, double-buffered so that the next K slice is read
// from global memory while the current one is multiplied.
template <typename TIn>
__global__ void __launch_bounds__(256) router_logits_kernel(const TIn* __restrict__ x,
                                                            const TIn* __restrict__ Wr,
                                                            const float* __restrict__ bias,
                                                            int T, int H, int E, int k_len,
                                                            float* __restrict__ out) {
  pdl_entry();
  constexpr int VEC = 16 / sizeof(TIn);                 // elements per 16-byte load
  constexpr int LOADS = RT_BM * RT_BK / VEC / 256;       // per thread per operand
  __shared__ __align__(16) float As[2][RT_BK][RT_BM + RT_PAD];
  __shared__ __align__(16) float Bs[2][RT_BK][RT_BN + RT_PAD];

  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int e0 = blockIdx.x * RT_BN, t0 = blockIdx.y * RT_BM;
  const int ks = blockIdx.z;
  const int kbeg = ks * k_len;
  const int kend = min(H, kbeg + k_len);

  unsigned long long acc[4][2];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = 0ull;

  float ra[LOADS][VEC], rb[LOADS][VEC];
  auto fetch = [&](int kb) {
#pragma unroll
    for (int l = 0; l < LOADS; ++l) {
      const int idx = tid + l * 256;
      const int row = idx % RT_BM;  // consecutive lanes -> consecutive rows
      const int kc = (idx / RT_BM) * VEC;
      const int t = t0 + row, e = e0 + row;
      if (t < T) {
        load_vec_f32<TIn>(x + (size_t)t * H + kb + kc, ra[l]);
      } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) ra[l][i] = 0.f;
      }
      if (e < E) {
        load_vec_f32<TIn>(Wr + (size_t)e * H + kb + kc, rb[l]);
      } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) rb[l][i] = 0.f;
      }
    }
  };
  auto stash = [&](int buf) {
#pragma unroll
    for (int l = 0; l < LOADS; ++l) {
      const int idx = tid + l * 256;
      const int row = idx % RT_BM;
      const int kc = (idx / RT_BM) * VEC;
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        As[buf][kc + i][row] = ra[l][i];
        Bs[buf][kc + i][row] = rb[l][i];
      }
    }
  };

  int buf = 0;
  if (kbeg < kend) {
    fetch(kbeg);
    stash(0);
  }
  __syncthreads();
  for (int kb = kbeg; kb < kend; kb += RT_BK) {
    const bool more = kb + RT_BK < kend;
    if (more) fetch(kb + RT_BK);
#pragma unroll
    for (int kk = 0; kk < RT_BK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
      const unsigned long long b01 = pack2(b.x, b.y), b23 = pack2(b.z, b.w);
      const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const unsigned long long ai = pack2(av[i], av[i]);
        fma2(acc[i][0], ai, b01);
        fma2(acc[i][1], ai, b23);
      }
    }
    if (more) stash(buf ^ 1);
    __syncthreads();
    buf ^= 1;
  }

  const bool add_bias = (bias != nullptr) && (gridDim.z == 1);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
    float v[4];
    unpack2(acc[i][0], v[0], v[1]);
    unpack2(acc[i][1], v[2], v[3]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e >= E) continue;
      float o = v[j];
      if (add_bias) o += bias[e];
      out[((size_t)ks * T + t) * E + e] = o;
    }
  }
}

// Large-batch variant: 128 tokens x 128 experts per CTA, 8 x 8 outputs per
// thread. Token values are stored twice in shared memory (x_t, x_t) so that a
// 16-byte load yields two ready fma.rn.f32x2 operands; expert weights are
// stored once and form (w_e, w_e+1) pairs. Per K step a thread issues six
// 16-byte shared loads for 64 FMAs (32 f32x2 instructions).
constexpr int RL_BM = 128, RL_BN = 128, RL_BK = 32;
constexpr int RL_APITCH = 2 * RL_BM + 8;   // floats per duplicated-token row
constexpr int RL_BPITCH = RL_BN + 4;       // floats per expert row
constexpr size_t RL_SMEM = sizeof(float) * 2 * RL_BK * (RL_APITCH + RL_BPITCH);

template <typename TIn>
__global__ void __launch_bounds__(256, 1) router_logits_big_kernel(
    const TIn* __restrict__ x, const TIn* __restrict__ Wr, const float* __restrict__ bias, int T,
    int H, int E, int k_len, float* __restrict__ out) {
  pdl_entry();
  constexpr int VEC = 16 / sizeof(TIn);
  constexpr int LOADS = RL_BM * RL_BK / VEC / 256;  // per thread per operand
  extern __shared__ __align__(16) float rl_sm[];
  float* As = rl_sm;                               // [2][BK][APITCH]
  float* Bs = rl_sm + 2 * RL_BK * RL_APITCH;       // [2][BK][BPITCH]

  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int e0 = blockIdx.x * RL_BN, t0 = blockIdx.y * RL_BM;
  const int ks = blockIdx.z;
  const int kbeg = ks * k_len;
  const int kend = min(H, kbeg + k_len);

  unsigned long long acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0ull;

  float ra[LOADS][VEC], rb[LOADS][VEC];
  auto fetch = [&](int kb) {
#pragma unroll
    for (int l = 0; l < LOADS; ++l) {
      const int idx = tid + l * 256;
      const int row = idx % RL_BM;
      const int kc = (idx / RL_BM) * VEC;
      const int t = t0 + row, e = e0 + row;
      if (t < T) {
        load_vec_f32<TIn>(x + (size_t)t * H + kb + kc, ra[l]);
      } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) ra[l][i] = 0.f;
      }
      if (e < E) {
        load_vec_f32<TIn>(Wr + (size_t)e * H + kb + kc, rb[l]);
      } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) rb[l][i] = 0.f;
      }
    }
  };
  auto stash = [&](int buf) {
    float* A = As + buf * RL_BK * RL_APITCH;
    float* B = Bs + buf * RL_BK * RL_BPITCH;
#pragma unroll
    for (int l = 0; l < LOADS; ++l) {
      const int idx = tid + l * 256;
      const int row = idx % RL_BM;
      const int kc = (idx / RL_BM) * VEC;
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        *reinterpret_cast<float2*>(&A[(kc + i) * RL_APITCH + 2 * row]) =
            make_float2(ra[l][i], ra[l][i]);
        B[(kc + i) * RL_BPITCH + row] = rb[l][i];
      }
    }
  };

  int buf = 0;
  if (kbeg < kend) {
    fetch(kbeg);
    stash(0);
  }
  __syncthreads();
  for (int kb = kbeg; kb < kend; kb += RL_BK) {
    const bool more = kb + RL_BK < kend;
    if (more) fetch(kb + RL_BK);
    const float* A = As + buf * RL_BK * RL_APITCH;
    const float* B = Bs + buf * RL_BK * RL_BPITCH;
#pragma unroll 4
    for (int kk = 0; kk < RL_BK; ++kk) {
      // tokens ty*8 .. ty*8+7 (duplicated pairs); experts tx*4..+3 and 64+tx*4..+3
      const ulonglong2* ap = reinterpret_cast<const ulonglong2*>(&A[kk * RL_APITCH + ty * 16]);
      const ulonglong2 a01 = ap[0], a23 = ap[1], a45 = ap[2], a67 = ap[3];
      const ulonglong2 b0 = *reinterpret_cast<const ulonglong2*>(&B[kk * RL_BPITCH + tx * 4]);
      const ulonglong2 b1 = *reinterpret_cast<const ulonglong2*>(&B[kk * RL_BPITCH + 64 + tx * 4]);
      const unsigned long long av[8] = {a01.x, a01.y, a23.x, a23.y, a45.x, a45.y, a67.x, a67.y};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        fma2(acc[i][0], av[i], b0.x);
        fma2(acc[i][1], av[i], b0.y);
        fma2(acc[i][2], av[i], b1.x);
        fma2(acc[i][3], av[i], b1.y);
      }
    }
    if (more) stash(buf ^ 1);
    __syncthreads();
    buf ^= 1;
  }

  const bool add_bias = (bias != nullptr) && (gridDim.z == 1);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + ty * 8 + i;
    if (t >= T) continue;
    float v[8];
    unpack2(acc[i][0], v[0], v[1]);
    unpack2(acc[i][1], v[2], v[3]);
    unpack2(acc[i][2], v[4], v[5]);
    unpack2(acc[i][3], v[6], v[7]);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = e0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
      if (e >= E) continue;
      float o = v[j];
      if (add_bias) o += bias[e];
      out[((size_t)ks * T + t) * E + e] = o;
    }
  }
}

// ---------------------------------------------------------------- tensor cores
// bf16 logits on tcgen05: one CTA per (128-token tile, expert tile of up to 256,
// slice of H). A = 128 token rows of x, B = n_tile expert rows of Wr, both
// K-major in 128-byte swizzled stages loaded by TMA; the 128 x n_tile fp32
// accumulator lives in TMEM (lane = token, column = expert). Token and expert
// tails read as zeros (TMA out-of-bounds fill) and are not stored.
constexpr int RC_BM = 128;          // tokens per tile (MMA M)
constexpr int RC_BK = 64;           // K per stage: one 128-byte row of bf16
constexpr int RC_MAX_N = 256;       // experts per tile (MMA N limit)
constexpr int RC_MAX_STAGES = 8;
constexpr int RC_RING_BYTES = 200 * 1024;

struct RouterTcArgs {
  CUtensorMap tmX;  // x [T][H], box 64 x 128 rows
  CUtensorMap tmW;  // Wr [E][H], box 64 x n_tile rows
  const float* bias;
  float* out;  // [S][T][E]
  int* status;
  unsigned long long limit_ns;
  int T, E, H, k_len, n_tile, stages, tmem_cols;
};

int rc_n_tile(int E) { return E >= RC_MAX_N ? RC_MAX_N : (E + 15) / 16 * 16; }
int rc_stage_bytes(int n_tile) { return RC_BM * 128 + n_tile * 128; }
int rc_stages(int n_tile) {
  const int s = RC_RING_BYTES / rc_stage_bytes(n_tile);
  return s > RC_MAX_STAGES ? RC_MAX_STAGES : s;
}
size_t rc_smem_bytes(int n_tile) {
  return 1024 /* alignment slack */ + (size_t)rc_stages(n_tile) * rc_stage_bytes(n_tile) +
         (2 * RC_MAX_STAGES + 1) * 8 + 16;
}

__global__ void __launch_bounds__(128, 1)
    router_logits_tc_kernel(const __grid_constant__ RouterTcArgs a) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int N = a.n_tile, ST = a.stages;
  const uint32_t A_BYTES = RC_BM * 128, STAGE = A_BYTES + (uint32_t)N * 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)ST * STAGE);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * RC_MAX_STAGES + 1);
  auto full_bar = [&](int i) { return smem_u32(&bars[i]); };
  auto empty_bar = [&](int i) { return smem_u32(&bars[RC_MAX_STAGES + i]); };
  const uint32_t done_bar = smem_u32(&bars[2 * RC_MAX_STAGES]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * RC_BM, e0 = blockIdx.y * N, slice = blockIdx.z;
  const int kbeg = slice * a.k_len;
  const int kend = min(a.H, kbeg + a.k_len);
  const int nk = (kend - kbeg) / RC_BK;  // H and k_len are multiples of RC_BK

  if (threadIdx.x == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 1);
    }
    mbar_init(done_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tmX);
    tma_prefetch_desc(&a.tmW);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), (uint32_t)a.tmem_cols);
  pdl_wait();  // global memory from here on
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol = l2_policy_evict_normal();
    int issued = 0;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % ST;
      const uint32_t round = (uint32_t)(kb / ST);
      if (!mbar_wait(empty_bar(s), (round & 1u) ^ 1u, a.status, a.limit_ns)) break;
      const uint32_t dst = smem_u32(smem + (size_t)s * STAGE);
      mbar_arrive_expect_tx(full_bar(s), STAGE);
      tma_load_2d(dst, &a.tmX, kbeg + kb * RC_BK, t0, full_bar(s), pol);
      tma_load_2d(dst + A_BYTES, &a.tmW, kbeg + kb * RC_BK, e0, full_bar(s), pol);
      ++issued;
    }
    // Let the last loads land before the CTA can exit (bounded, status ignored).
    const int n_last = issued < ST ? issued : ST;
    for (int i = issued - n_last; i < issued; ++i)
      mbar_wait(full_bar(i % ST), (uint32_t)(i / ST) & 1u, nullptr, 20000000ull);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = umma_idesc(1u, RC_BM, (uint32_t)N);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % ST;
      const uint32_t round = (uint32_t)(kb / ST);
      if (!mbar_wait(full_bar(s), round & 1u, a.status, a.limit_ns)) break;
      tc_fence_after();
      const uint32_t a_addr = smem_u32(smem + (size_t)s * STAGE);
      const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
      for (int kk = 0; kk < RC_BK / 16; ++kk)
        umma_issue<kKindF16>(tmem, umma_desc_sw128(a_addr + kk * 32),
                          umma_desc_sw128(b_addr + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
      umma_commit(empty_bar(s));
    }
    // Arrives once every MMA issued above has completed (also after a timeout).
    umma_commit(done_bar);
  }
  __syncwarp();

  // -------------------------------------------------------------- epilogue
  // Warp w reads TMEM lanes 32w..32w+31 (tokens); 32 expert columns per load.
  bool ok = mbar_wait(done_bar, 0, a.status, a.limit_ns) && read_status(a.status) == MOE_OK;
  ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-collective
  if (ok) {
    tc_fence_after();
    const int t = t0 + warp * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
    float* orow = a.out + ((size_t)slice * a.T + (size_t)(t < a.T ? t : 0)) * a.E;
    const float* bias = (a.bias != nullptr && gridDim.z == 1) ? a.bias : nullptr;
    const bool vec = (a.E & 3) == 0;
    for (int c0 = 0; c0 < N; c0 += 32) {
      float v[32];
      tmem_ld32(taddr + (uint32_t)c0, v);
      const int eb = e0 + c0;
      if (t < a.T) {
        if (vec && eb + 32 <= a.E) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            float4 o = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
            if (bias) {
              o.x += bias[eb + i];
              o.y += bias[eb + i + 1];
              o.z += bias[eb + i + 2];
              o.w += bias[eb + i + 3];
            }
            *reinterpret_cast<float4*>(orow + eb + i) = o;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (eb + i < a.E) orow[eb + i] = bias ? v[i] + bias[eb + i] : v[i];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
  }
}

cudaError_t launch_router_logits_tc(const void* x, const void* Wr, const float* bias, int T,
                                    int H, int E, int S, int k_len, float* out, int* status,
                                    unsigned long long limit_ns, cudaStream_t st) {
  RouterTcArgs a;
  memset(&a, 0, sizeof(a));
  const int n_tile = rc_n_tile(E);
  if (!make_tma_map(&a.tmX, x, MOE_DTYPE_BF16, (uint64_t)T, (uint64_t)H, RC_BM) ||
      !make_tma_map(&a.tmW, Wr, MOE_DTYPE_BF16, (uint64_t)E, (uint64_t)H, (uint32_t)n_tile))
    return cudaErrorInvalidValue;
  a.bias = bias;
  a.out = out;
  a.status = status;
  a.limit_ns = limit_ns;
  a.T = T;
  a.E = E;
  a.H = H;
  a.k_len = k_len;
  a.n_tile = n_tile;
  a.stages = rc_stages(n_tile);
  int cols = 32;
  while (cols < n_tile) cols *= 2;
  a.tmem_cols = cols;
  const size_t smem = rc_smem_bytes(n_tile);
  // Opt in once per device for the largest ring (any n_tile fits under it).
  static std::mutex mu;
  static bool opted[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64 || !opted[dev]) {
      e = cudaFuncSetAttribute(router_logits_tc_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)(RC_RING_BYTES + 4096));
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) opted[dev] = true;
    }
  }
  dim3 grid((unsigned)((T + RC_BM - 1) / RC_BM), (unsigned)((E + n_tile - 1) / n_tile),
            (unsigned)S);
  return launch_chained(router_logits_tc_kernel, grid, dim3(128), smem, st, 1, a);
}

// Sum of S partial logits in ascending slice order, then the bias: identical
// arithmetic in the reduction kernel and in the route kernel.
// The loads of each batch of 8 slices are issued together (they are
// independent); the additions keep ascending slice order.
__device__ __forceinline__ float reduce_partials(const float* __restrict__ part, int S, int T,
                                                 int E, int t, int e,
                                                 const float* __restrict__ bias) {
  const size_t stride = (size_t)T * E;
  const float* p = part + (size_t)t * E + e;
  float v = p[0];
  int s = 1;
  for (; s + 8 <= S; s += 8) {
    float q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = p[(size_t)(s + j) * stride];
#pragma unroll
    for (int j = 0; j < 8; ++j) v += q[j];
  }
  for (; s < S; ++s) v += p[(size_t)s * stride];
  if (bias) v += bias[e];
  return v;
}

__global__ void logits_reduce_kernel(const float* __restrict__ part, int S, int T, int E,
                                     const float* __restrict__ bias, float* __restrict__ logits) {
  pdl_entry();
  const size_t n = (size_t)T * E;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / E), e = (int)(i % E);
    logits[i] = reduce_partials(part, S, T, E, t, e, bias);
  }
}

// S == 1: `src` holds final logits (bias already added). S > 1: `src` holds S
// partial slices; they are reduced here and, if logits_out != nullptr, the
// reduced logits are written out.
// B: partial slices loaded together (all of a batch's loads are issued before
// any of them is added). One-slice batches need the fewest registers and suit
// S <= 2; larger batches cut the dependent load round trips when S is larger.
template <int NV, int B>
__global__ void __launch_bounds__(256, 2) route_kernel(const float* __restrict__ src, int S,
                                                    const float* __restrict__ bias, int T, int E,
                                                    int k, int renorm, int n_group,
                                                    int topk_group,
                                                    float* __restrict__ logits_out,
                                                    int32_t* __restrict__ ids,
                                                    float* __restrict__ w) {
  pdl_entry();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  float v[NV];
  const float* row = src + (size_t)t * E;
  if (S == 1) {
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? row[e] : -INFINITY;
    }
  } else {
    // Sum of the S partial slices in ascending slice order, then the bias (the
    // arithmetic of reduce_partials).
    const size_t stride = (size_t)T * E;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? row[e] : 0.f;
    }
    for (int s0 = 1; s0 < S; s0 += B) {
      float q[NV][B];
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
#pragma unroll
        for (int j = 0; j < B; ++j)
          q[i][j] = (e < E && s0 + j < S) ? row[(size_t)(s0 + j) * stride + e] : 0.f;
      }
#pragma unroll
      for (int i = 0; i < NV; ++i)
#pragma unroll
        for (int j = 0; j < B; ++j)
          if (s0 + j < S) v[i] += q[i][j];
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        if (bias) v[i] += bias[e];
        if (logits_out) logits_out[(size_t)t * E + e] = v[i];
      } else {
        v[i] = -INFINITY;
      }
    }
  }
  route_warp<NV>(v, E, k, renorm, n_group, topk_group, ids + (size_t)t * k, w + (size_t)t * k);
}

}  // namespace

// Batches of at least this many tokens use the 128 x 128 tile kernel.
constexpr int64_t kRouterBigT = 1024;

int64_t router_split_request(int64_t T, int64_t H, int64_t E, int num_sms);

// K step of each router kernel: slices of H are multiples of it.
int64_t router_k_step(int dtype) { return dtype == MOE_DTYPE_BF16 ? RC_BK : RT_BK; }

// Slice length for S slices of H: a multiple of the K step.
int64_t router_slice_len(int dtype, int64_t H, int64_t S) {
  const int64_t step = router_k_step(dtype);
  const int64_t k_len = (H + S - 1) / S;
  return (k_len + step - 1) / step * step;
}

// Slices actually produced by S requested slices (rounding the slice length
// up can leave fewer).
int64_t router_effective_slices(int dtype, int64_t H, int64_t S) {
  const int64_t k_len = router_slice_len(dtype, H, S);
  return (H + k_len - 1) / k_len;
}

// Tensor-core split: as many slices as fill one wave of one CTA per SM, each
// at least two stages (128) of H long, and at most kRouterMaxSlices: the route
// kernel adds the slices, and more than a few of them cost it more latency
// than they save here.
constexpr int64_t kRouterMaxSlices = 8;
int64_t router_tc_split_request(int64_t T, int64_t H, int64_t E, int num_sms) {
  const int64_t n_tile = rc_n_tile((int)E);
  const int64_t tiles = ((T + RC_BM - 1) / RC_BM) * ((E + n_tile - 1) / n_tile);
  if (tiles <= 0) return 1;
  int64_t smax = H / (2 * RC_BK) < 1 ? 1 : H / (2 * RC_BK);
  if (smax > kRouterMaxSlices) smax = kRouterMaxSlices;
  const int64_t S = num_sms / tiles;
  return S < 1 ? 1 : (S > smax ? smax : S);
}

int router_split_count(int dtype, int64_t T, int64_t H, int64_t E, int num_sms) {
  const int64_t req = dtype == MOE_DTYPE_BF16 ? router_tc_split_request(T, H, E, num_sms)
                                              : router_split_request(T, H, E, num_sms);
  return (int)router_effective_slices(dtype, H, req);
}

int64_t router_split_request(int64_t T, int64_t H, int64_t E, int num_sms) {
  const bool big = T >= kRouterBigT;
  const int64_t bm = big ? RL_BM : RT_BM, bn = big ? RL_BN : RT_BN;
  const int64_t resident = (big ? 1 : 4) * (int64_t)num_sms;  // CTAs per wave
  const int64_t tiles = ((E + bn - 1) / bn) * ((T + bm - 1) / bm);
  if (tiles <= 0) return 1;
  const int64_t smax = H / 128 < 1 ? 1 : H / 128;  // at least 128 of H per slice
  if (!big) {
    int64_t S = (resident + tiles - 1) / tiles;
    return (int)(S > smax ? smax : (S < 1 ? 1 : S));
  }
  // Smallest split whose last wave is at least 90% full (at most 8 slices),
  // else the best-filled one.
  int64_t best = 1;
  double best_eff = 0.0;
  for (int64_t S = 1; S <= 8 && S <= smax; ++S) {
    const double waves = (double)(tiles * S) / (double)resident;
    const double eff = waves / std::ceil(waves);
    if (eff >= 0.9) return (int)S;
    if (eff > best_eff) {
      best_eff = eff;
      best = S;
    }
  }
  return (int)best;
}

cudaError_t launch_router_logits(int dtype, const void* x, const void* Wr, const float* bias,
                                 int T, int H, int E, int S, float* out_partials, int* status,
                                 unsigned long long limit_ns, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int k_len = (int)router_slice_len(dtype, H, S);
  if (router_effective_slices(dtype, H, S) != S) return cudaErrorInvalidValue;
  if (dtype == MOE_DTYPE_BF16)
    return launch_router_logits_tc(x, Wr, bias, T, H, E, S, k_len, out_partials, status,
                                   limit_ns, st);
  if (T >= kRouterBigT) {
    dim3 grid((E + RL_BN - 1) / RL_BN, (T + RL_BM - 1) / RL_BM, S);
    cudaError_t e;
    if (dtype == MOE_DTYPE_BF16) {
      e = cudaFuncSetAttribute(router_logits_big_kernel<__nv_bfloat16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RL_SMEM);
      if (e != cudaSuccess) return e;
      return launch_chained(router_logits_big_kernel<__nv_bfloat16>, grid, dim3(256),
                            (size_t)RL_SMEM, st, 1, (const __nv_bfloat16*)x,
                            (const __nv_bfloat16*)Wr, bias, T, H, E, k_len, out_partials);
    } else {
      e = cudaFuncSetAttribute(router_logits_big_kernel<float>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RL_SMEM);
      if (e != cudaSuccess) return e;
      return launch_chained(router_logits_big_kernel<float>, grid, dim3(256), (size_t)RL_SMEM,
                            st, 1, (const float*)x, (const float*)Wr, bias, T, H, E, k_len,
                            out_partials);
    }
  }
  dim3 grid((E + RT_BN - 1) / RT_BN, (T + RT_BM - 1) / RT_BM, S);
  if (dtype == MOE_DTYPE_BF16)
    return launch_chained(router_logits_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, 1,
                          (const __nv_bfloat16*)x, (const __nv_bfloat16*)Wr, bias, T, H, E, k_len,
                          out_partials);
  return launch_chained(router_logits_kernel<float>, grid, dim3(256), 0, st, 1, (const float*)x,
                        (const float*)Wr, bias, T, H, E, k_len, out_partials);
}

cudaError_t launch_logits_reduce(const float* partials, int S, int T, int E, const float* bias,
                                 float* logits, int num_sms, cudaStream_t st) {
  const size_t n = (size_t)T * E;
  if (n == 0) return cudaSuccess;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 8 * num_sms) blocks = 8 * num_sms;
  return launch_chained(logits_reduce_kernel, dim3(blocks), dim3(256), 0, st, 1, partials, S, T,
                        E, bias, logits);
}

cudaError_t launch_route(const float* src, int S, const float* bias, int T, int E, int k,
                         int renorm, int n_group, int topk_group, float* logits_out,
                         int32_t* ids, float* w, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int warps = 8;
  const int blocks = (T + warps - 1) / warps;
  const int nv = (E + 31) / 32;
  // Batches of 32 / NV slices (one load round trip for up to 8 slices when
  // NV <= 4) unless at most one slice is added to the first.
  const bool wide = S > 2;
#define MOE_ROUTE_CASE(NV)                                                                     \
  return wide ? launch_chained(route_kernel<NV, (NV >= 32 ? 1 : 32 / NV)>, dim3(blocks),      \
                               dim3(warps * 32), 0, st, 1, src, S, bias, T, E, k, renorm,      \
                               n_group, topk_group, logits_out, ids, w)                        \
              : launch_chained(route_kernel<NV, 1>, dim3(blocks), dim3(warps * 32), 0, st, 1, \
                               src, S, bias, T, E, k, renorm, n_group, topk_group, logits_out, \
                               ids, w)
  if (nv <= 1) MOE_ROUTE_CASE(1);
  else if (nv <= 2) MOE_ROUTE_CASE(2);
  else if (nv <= 4) MOE_ROUTE_CASE(4);
  else if (nv <= 8) MOE_ROUTE_CASE(8);
  else if (nv <= 16) MOE_ROUTE_CASE(16);
  else MOE_ROUTE_CASE(32);
#undef MOE_ROUTE_CASE
  return cudaGetLastError();
}

}  // namespace moe
