// MXFP8 block quantization: the expert weights of the MXFP8 layer (once) and
// its token rows x (each forward).
//
// "Hosting Qwen on Blackwell" (quantization section) serves Qwen3-235B with
// MXFP8 weights converted statically; "CuTeDSL at Perplexity" (Blackwell
// quantization paragraph) computes MXFP8 scales from the absolute maximum over
// 32 elements. The block rule is the Microscaling format's: per block of 32
// consecutive elements along a row,
//   e = floor(log2(amax)) - 8 (8: exponent of E4M3's largest power of two),
//       held in [-127, 127]; e = -127 for a block of zeros;
//   scale byte = e + 127 (E8M0), codes = E4M3(v * 2^-e), nearest even,
//   saturating at 448 (the block's largest element scales into [256, 512)).
// Scaling by 2^-e is exact in fp32 (no flush of subnormals in this build), so
// the only rounding is the conversion of each element. One thread per block.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"
#include "mx.cuh"

namespace moe {

namespace {

__device__ __forceinline__ void load32(const __nv_bfloat16* p, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = reinterpret_cast<const uint4*>(p)[i];
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(b[j]);
      v[8 * i + 2 * j] = f.x;
      v[8 * i + 2 * j + 1] = f.y;
    }
  }
}

__device__ __forceinline__ void load32(const float* p, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 a = reinterpret_cast<const float4*>(p)[i];
    v[4 * i] = a.x;
    v[4 * i + 1] = a.y;
    v[4 * i + 2] = a.z;
    v[4 * i + 3] = a.w;
  }
}

// Thread = one scale byte of one row: blocks b < cols / 32 are quantized,
// b in [cols / 32, sk) is the row's zero padding. QDQ: instead of codes and
// scales, the bf16 value of every element after quantization is written to
// out (x of the MXFP8 layer, which its GEMMs read as bf16).
template <typename TIn, bool QDQ>
__global__ void __launch_bounds__(256) quantize_mx_kernel(const TIn* __restrict__ src,
                                                          int64_t rows, int cols, int sk,
                                                          uint8_t* __restrict__ q,
                                                          uint8_t* __restrict__ scales,
                                                          __nv_bfloat16* __restrict__ out) {
  pdl_entry();
  const int nb = cols / 32;
  const int per_row = QDQ ? nb : sk;
  const int64_t n = rows * per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / per_row;
    const int b = (int)(i - r * per_row);
    if (!QDQ && b >= nb) {
      scales[r * sk + b] = 0;
      continue;
    }
    const int64_t off = r * cols + (int64_t)b * 32;
    float v[32];
    load32(src + off, v);
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
    const int e = mx_block_exponent(amax);
    const float inv = mx_pow2(-e);
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = mx_encode4(v[4 * j] * inv, v[4 * j + 1] * inv,
                                                  v[4 * j + 2] * inv, v[4 * j + 3] * inv);
    if constexpr (QDQ) {
      const float X = mx_pow2(e);
      uint32_t o[16];
#pragma unroll
      for (int j = 0; j < 8; ++j) mx_decode4_bf16(w[j], X, o[2 * j], o[2 * j + 1]);
      uint4* dst = reinterpret_cast<uint4*>(out + off);
#pragma unroll
      for (int j = 0; j < 4; ++j) dst[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
    } else {
      uint4* dst = reinterpret_cast<uint4*>(q + off);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      scales[r * sk + b] = (uint8_t)(e + 127);
    }
  }
}

// The MXFP8 decode-sized layer's token operand in one pass: warp = routed
// slot s (token s / k), lane = one block of 32 elements per step. The slot's
// codes and scale row go to row slot_pos[s] of xgq / xgs (the expert-ordered
// copy the GEMMs read as tiles); the token's first slot also writes row t of
// xq / xs (token order, for the shared expert) when those are given. A
// position beyond T*k sets MOE_ERR_DEVICE_CHECK and the slot is skipped.
__global__ void __launch_bounds__(256) quantize_dispatch_mx_kernel(
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ slot_pos, int T, int k,
    int H, int sk, uint8_t* __restrict__ xgq, uint8_t* __restrict__ xgs, uint8_t* __restrict__ xq,
    uint8_t* __restrict__ xs, int* status) {
  pdl_entry();
  const int lane = threadIdx.x & 31;
  const int P = T * k;
  const int nb = H / 32;
  const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t s = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; s < P; s += warps) {
    const int p = slot_pos[s];
    if ((unsigned)p >= (unsigned)P) {
      if (lane == 0) set_status(status, MOE_ERR_DEVICE_CHECK);
      continue;
    }
    const int t = (int)(s / k);
    const bool token_row = xq != nullptr && s - (int64_t)t * k == 0;
    for (int b = lane; b < sk; b += 32) {
      if (b >= nb) {  // the scale row's padding
        xgs[(size_t)p * sk + b] = 0;
        if (token_row) xs[(size_t)t * sk + b] = 0;
        continue;
      }
      float v[32];
      load32(x + (size_t)t * H + (size_t)b * 32, v);
      float amax = 0.0f;
#pragma unroll
      for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
      const int e = mx_block_exponent(amax);
      const float inv = mx_pow2(-e);
      uint32_t w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        w[j] = mx_encode4(v[4 * j] * inv, v[4 * j + 1] * inv, v[4 * j + 2] * inv,
                          v[4 * j + 3] * inv);
      uint4* dst = reinterpret_cast<uint4*>(xgq + (size_t)p * H + (size_t)b * 32);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      xgs[(size_t)p * sk + b] = (uint8_t)(e + 127);
      if (token_row) {
        uint4* dt = reinterpret_cast<uint4*>(xq + (size_t)t * H + (size_t)b * 32);
        dt[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dt[1] = make_uint4(w[4], w[5], w[6], w[7]);
        xs[(size_t)t * sk + b] = (uint8_t)(e + 127);
      }
    }
  }
}

unsigned grid_for(int64_t n, int num_sms) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > 16 * (int64_t)num_sms) blocks = 16 * (int64_t)num_sms;
  return (unsigned)(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_quantize_mx(int dtype, const void* src, int64_t rows, int64_t cols,
                               uint8_t* q, uint8_t* scales, int num_sms, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int sk = mx_scale_cols((int)cols);
  const unsigned g = grid_for(rows * sk, num_sms);
  if (dtype == MOE_DTYPE_BF16)
    return launch_chained(quantize_mx_kernel<__nv_bfloat16, false>, dim3(g), dim3(256), 0, st, 1,
                          (const __nv_bfloat16*)src, rows, (int)cols, sk, q, scales,
                          (__nv_bfloat16*)nullptr);
  return launch_chained(quantize_mx_kernel<float, false>, dim3(g), dim3(256), 0, st, 1,
                        (const float*)src, rows, (int)cols, sk, q, scales,
                        (__nv_bfloat16*)nullptr);
}

cudaError_t launch_quantize_dispatch_mx(const void* x, const int32_t* slot_pos, int T, int k,
                                       int H, uint8_t* xgq, uint8_t* xgs, uint8_t* xq, uint8_t* xs,
                                       int* status, int num_sms, cudaStream_t st) {
  const int P = T * k;
  if (P == 0) return cudaSuccess;
  int64_t blocks = ((int64_t)P + 7) / 8;
  if (blocks > 16 * (int64_t)num_sms) blocks = 16 * (int64_t)num_sms;
  return launch_chained(quantize_dispatch_mx_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1,
                        (const __nv_bfloat16*)x, slot_pos, T, k, H, mx_scale_cols(H), xgq, xgs,
                        xq, xs, status);
}

cudaError_t launch_qdq_mx(const void* src, int64_t rows, int64_t cols, void* out, int num_sms,
                          cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const unsigned g = grid_for(rows * (cols / 32), num_sms);
  return launch_chained(quantize_mx_kernel<__nv_bfloat16, true>, dim3(g), dim3(256), 0, st, 1,
                        (const __nv_bfloat16*)src, rows, (int)cols, 0, (uint8_t*)nullptr,
                        (uint8_t*)nullptr, (__nv_bfloat16*)out);
}

}  // namespace moe
