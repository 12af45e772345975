// Row quantization to E4M3 with one power-of-two scale per row: the FP8
// expert path's weights (once), token rows x and hidden rows h (each forward).
//
// Microscaling as "Hosting Qwen on Blackwell" describes it for Blackwell's FP8
// serving: the scale factor is a power of two, so scaling never rounds and the
// only rounding is the conversion of each element to E4M3. Per row r:
//   e = the smallest integer with max_i |v_i| <= 448 * 2^e (448 = 1.75 * 2^8 is
//       the largest finite E4M3 magnitude), at least -126; e = 0 for a zero row;
//   scale[r] = 2^e, q[r][i] = E4M3(v_i * 2^-e), nearest, ties to even.
// Dequantization is q * scale. One warp per row: an absolute-maximum reduction,
// then the scaled conversion (the row is read twice; the second read hits L1).
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

// e of the rule above from the bits of amax: amax = (1 + f) * 2^E with
// f = frac / 2^23; 1 + f <= 1.75 exactly when frac <= 0x600000.
__device__ __forceinline__ int row_exponent(float amax) {
  if (!(amax > 0.0f)) return 0;
  const uint32_t b = __float_as_uint(amax);
  const int ef = (int)((b >> 23) & 0xFFu);
  if (ef == 0) return -126;  // subnormal maximum: the floor applies
  const int E = ef - 127;
  const int e = (b & 0x7FFFFFu) <= 0x600000u ? E - 8 : E - 7;
  return e < -126 ? -126 : e;
}

__device__ __forceinline__ float pow2(int e) {  // e in [-126, 127]
  return __uint_as_float((uint32_t)(e + 127) << 23);
}

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(b[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Eight consecutive elements per lane and step; cols is a multiple of 16.
template <typename TIn>
__global__ void __launch_bounds__(256) quantize_rows_kernel(const TIn* __restrict__ src,
                                                            int64_t rows, int cols,
                                                            uint8_t* __restrict__ q,
                                                            float* __restrict__ scale) {
  pdl_entry();
  const int lane = threadIdx.x & 31;
  const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
    const TIn* row = src + r * cols;
    float amax = 0.0f;
    for (int c = lane * 8; c < cols; c += 256) {
      float v[8];
      load8(row + c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const int e = row_exponent(amax);
    const float inv = pow2(-e);  // -e in [-120, 126]: exact multiply
    uint8_t* qrow = q + r * cols;
    for (int c = lane * 8; c < cols; c += 256) {
      float v[8];
      load8(row + c, v);
      uint32_t w[2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_fp8x2_storage_t p2 = __nv_cvt_float2_to_fp8x2(
            make_float2(v[2 * i] * inv, v[2 * i + 1] * inv), __NV_SATFINITE, __NV_E4M3);
        if (i % 2 == 0)
          w[i / 2] = (uint32_t)p2;
        else
          w[i / 2] |= (uint32_t)p2 << 16;
      }
      *reinterpret_cast<uint2*>(qrow + c) = make_uint2(w[0], w[1]);
    }
    if (lane == 0) scale[r] = pow2(e);
  }
}

}  // namespace

cudaError_t launch_quantize_rows(int dtype, const void* src, int64_t rows, int64_t cols,
                                 uint8_t* q, float* scale, int num_sms, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  int64_t blocks = (rows + 7) / 8;
  if (blocks > 16 * (int64_t)num_sms) blocks = 16 * (int64_t)num_sms;
  if (dtype == MOE_DTYPE_BF16)
    return launch_chained(quantize_rows_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256),
                          0, st, 1, (const __nv_bfloat16*)src, rows, (int)cols, q, scale);
  return launch_chained(quantize_rows_kernel<float>, dim3((unsigned)blocks), dim3(256), 0, st, 1,
                        (const float*)src, rows, (int)cols, q, scale);
}

}  // namespace moe
