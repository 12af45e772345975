// MXFP8 element and scale helpers shared by the quantization kernels and the
// MXFP8 grouped GEMM (blocks of 32 E4M3 codes with one E8M0 scale byte).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace moe {

// Scale bytes per row of `cols` elements: one per block of 32, the row padded
// to a multiple of 16 bytes (a TMA row stride).
__host__ __device__ constexpr int mx_scale_cols(int cols) { return 16 * ((cols / 32 + 15) / 16); }

// 2^e as fp32, e in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float mx_pow2(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23)
                   : __uint_as_float(1u << (e + 149));
}

// Block exponent: floor(log2(amax)) - 8, held at -127 from below; -127 for a
// block of zeros. amax is finite and >= 0; its floor(log2) is read from the
// bits (subnormals included), so it is exact.
__device__ __forceinline__ int mx_block_exponent(float amax) {
  if (!(amax > 0.0f)) return -127;
  const uint32_t b = __float_as_uint(amax);
  const int ef = (int)(b >> 23);
  const int fl = ef == 0 ? (31 - __clz((int)(b & 0x7FFFFFu))) - 149 : ef - 127;
  const int e = fl - 8;
  return e < -127 ? -127 : e;
}

// Four values -> four E4M3 codes (nearest even, saturating at 448), in memory
// order (the first value in the lowest byte).
__device__ __forceinline__ uint32_t mx_encode4(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE,
                                                           __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE,
                                                           __NV_E4M3);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Two E4M3 codes (low byte first) times X -> a bf16 pair (the first value in
// the low half), rounded to nearest even. The code converts exactly to fp16
// and fp32, and X is a power of two, so the only rounding is the final one
// (none for scales >= 2^-117, whose values are bf16 normals).
__device__ __forceinline__ uint32_t mx_decode2_bf16(uint32_t codes2, float X) {
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(codes2 & 0xFFFFu),
                                                    __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * X, f.y * X);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// Four codes -> two bf16 pairs (codes 0,1 in lo; 2,3 in hi).
__device__ __forceinline__ void mx_decode4_bf16(uint32_t codes4, float X, uint32_t& lo,
                                                uint32_t& hi) {
  lo = mx_decode2_bf16(codes4, X);
  hi = mx_decode2_bf16(codes4 >> 16, X);
}

// The scale 2^(byte - 127) of an E8M0 byte.
__device__ __forceinline__ float mx_scale_of(uint32_t byte) { return mx_pow2((int)byte - 127); }

}  // namespace moe
