// The rank-order combine of the down projection's slot rows for the
// single-launch decode kernel (fused_decode.cu): the reduction of the combine
// kernel in combine.cu, as a device function over a range of items. The
// stand-alone kernel keeps its own copy of the loop: compiled through this
// function it measured 5% slower at the prefill chunk's size.
#pragma once

#include "common.cuh"

namespace moe {

// y[t][c] = sum_{j < KP} Y[t][j][c] in fp32, rank order j = 0..KP-1, one
// rounding to TOut; four consecutive features per item, items i0, i0 + step,
// ... below T * H / 4. Y is read with streaming loads (each slot is read once).
template <typename TOut>
__device__ __forceinline__ void combine_range(const float* __restrict__ Y, int T, int H, int KP,
                                              TOut* __restrict__ y, size_t i0, size_t step) {
  const int h4 = H / 4;
  const size_t n = (size_t)T * h4;
  for (size_t i = i0; i < n; i += step) {
    const size_t t = i / h4;
    const int c4 = (int)(i - t * h4);
    const float4* src = reinterpret_cast<const float4*>(Y + t * KP * H) + c4;
    float4 a = __ldcs(src);
    for (int j = 1; j < KP; ++j) {
      const float4 b = __ldcs(src + (size_t)j * h4);
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    if constexpr (sizeof(TOut) == 2) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(a.z, a.w);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&lo);
      pk.y = *reinterpret_cast<const uint32_t*>(&hi);
      reinterpret_cast<uint2*>(y + t * H)[c4] = pk;
    } else {
      reinterpret_cast<float4*>(y + t * H)[c4] = a;
    }
  }
}

}  // namespace moe
