// Router: logits (step a1) and top-k routing with gate weights (step a2).
//
// Logits: logits[t][e] = sum_h x[t][h] * Wr[e][h] (+ b[e]) with fp32
// accumulation on the CUDA cores ("Gate" at the end of stage 2 of the
// five-stage MoE layer in "Lower latency and higher throughput with multi-node
// DeepSeek deployment"). When the tile grid alone cannot fill the GPU (decode:
// T = 64), H is split into S slices whose partial sums are added later in
// ascending slice order, so results do not depend on scheduling.
//
// Route: one warp per token keeps the token's E logits in registers, takes the
// k largest one at a time (lowest expert index among equal values), then the
// softmax gate weights over the chosen k (renorm) or over all E ("MoE Router"
// section of the same page: top-k indices and scores per token).
#include "common.cuh"
#include "kernels.h"

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

// Sum of S partial logits in ascending slice order, then the bias: identical
// arithmetic in the reduction kernel and in the route kernel.
__device__ __forceinline__ float reduce_partials(const float* __restrict__ part, int S, int T,
                                                 int E, int t, int e,
                                                 const float* __restrict__ bias) {
  float v = part[(size_t)t * E + e];
  for (int s = 1; s < S; ++s) v += part[((size_t)s * T + t) * E + e];
  if (bias) v += bias[e];
  return v;
}

__global__ void logits_reduce_kernel(const float* __restrict__ part, int S, int T, int E,
                                     const float* __restrict__ bias, float* __restrict__ logits) {
  const size_t n = (size_t)T * E;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / E), e = (int)(i % E);
    logits[i] = reduce_partials(part, S, T, E, t, e, bias);
  }
}

// One warp per token. NV = values per lane (E <= 32 * NV).
// S == 1: `src` holds final logits (bias already added). S > 1: `src` holds S
// partial slices; they are reduced here and, if logits_out != nullptr, the
// reduced logits are written out.
template <int NV>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ src, int S,
                                                    const float* __restrict__ bias, int T, int E,
                                                    int k, int renorm,
                                                    float* __restrict__ logits_out,
                                                    int32_t* __restrict__ ids,
                                                    float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;

  float v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      v[i] = (S == 1) ? src[(size_t)t * E + e] : reduce_partials(src, S, T, E, t, e, bias);
      if (S > 1 && logits_out) logits_out[(size_t)t * E + e] = v[i];
    } else {
      v[i] = -INFINITY;
    }
  }

  // k rounds of warp arg-max over the not-yet-chosen values; ties go to the
  // lower expert index. Lane r keeps round r's (value, index).
  uint32_t taken = 0;
  float my_val = 0.f;
  int my_idx = 0;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      const bool free_ = !((taken >> i) & 1u) && e < E;
      if (free_ && (v[i] > bv || bi == 0x7fffffff)) {  // ascending e: first max wins
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == r) {
      my_val = bv;
      my_idx = bi;
    }
  }

  const float m = __shfl_sync(0xffffffffu, my_val, 0);
  float p = (lane < k) ? expf(my_val - m) : 0.f;
  float ssum;
  if (renorm) {
    ssum = p;
  } else {
    ssum = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (lane + 32 * i < E) ssum += expf(v[i] - m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, off);
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_idx;
    w[(size_t)t * k + lane] = p / ssum;
  }
}

}  // namespace

int router_split_count(int64_t T, int64_t H, int64_t E, int num_sms) {
  const int64_t tiles = ((E + RT_BN - 1) / RT_BN) * ((T + RT_BM - 1) / RT_BM);
  if (tiles <= 0) return 1;
  // About four CTAs per SM in total, so the last wave is a small fraction.
  int64_t S = (4 * (int64_t)num_sms + tiles - 1) / tiles;
  const int64_t smax = H / 128;  // at least 128 of H per slice
  if (S > smax) S = smax;
  if (S < 1) S = 1;
  return (int)S;
}

cudaError_t launch_router_logits(int dtype, const void* x, const void* Wr, const float* bias,
                                 int T, int H, int E, int S, float* out_partials,
                                 cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  int k_len = (H + S - 1) / S;
  k_len = (k_len + RT_BK - 1) / RT_BK * RT_BK;
  const int S_eff = (H + k_len - 1) / k_len;
  if (S_eff != S) return cudaErrorInvalidValue;
  dim3 grid((E + RT_BN - 1) / RT_BN, (T + RT_BM - 1) / RT_BM, S);
  if (dtype == MOE_DTYPE_BF16) {
    router_logits_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
        (const __nv_bfloat16*)x, (const __nv_bfloat16*)Wr, bias, T, H, E, k_len, out_partials);
  } else {
    router_logits_kernel<float>
        <<<grid, 256, 0, st>>>((const float*)x, (const float*)Wr, bias, T, H, E, k_len,
                               out_partials);
  }
  return cudaGetLastError();
}

int router_split_len_ok(int H, int S) {
  int k_len = (H + S - 1) / S;
  k_len = (k_len + RT_BK - 1) / RT_BK * RT_BK;
  return ((H + k_len - 1) / k_len) == S;
}

cudaError_t launch_logits_reduce(const float* partials, int S, int T, int E, const float* bias,
                                 float* logits, int num_sms, cudaStream_t st) {
  const size_t n = (size_t)T * E;
  if (n == 0) return cudaSuccess;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 8 * num_sms) blocks = 8 * num_sms;
  logits_reduce_kernel<<<blocks, 256, 0, st>>>(partials, S, T, E, bias, logits);
  return cudaGetLastError();
}

cudaError_t launch_route(const float* src, int S, const float* bias, int T, int E, int k,
                         int renorm, float* logits_out, int32_t* ids, float* w,
                         cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int warps = 8;
  const int blocks = (T + warps - 1) / warps;
  const int nv = (E + 31) / 32;
#define MOE_ROUTE_CASE(NV)                                                                  \
  route_kernel<NV><<<blocks, warps * 32, 0, st>>>(src, S, bias, T, E, k, renorm, logits_out, \
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
