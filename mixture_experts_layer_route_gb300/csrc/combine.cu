// Combine (the reduction half of step a5): y[t][c] = sum_{j < KP} Y[t][j][c],
// summed in rank order j = 0..k-1, then the shared-expert slot j = k. The
// gate weights were applied by the down-projection epilogue that wrote Y.
// "CuTeDSL at Perplexity", "Local" combine: a vectorised accumulation over the
// token's expert outputs; "Expert Parallelism" section of the DeepSeek page:
// weighted sum of the routed experts plus the shared expert.
//
// Pure streaming: 16-byte loads of the fp32 slots, one rounding to the output
// dtype, grid sized to a multiple of the SM count.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

template <typename TOut>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ Y, int T, int H,
                                                      int KP, TOut* __restrict__ y) {
  pdl_entry();
  const int h4 = H / 4;
  const size_t n = (size_t)T * h4;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
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

}  // namespace

cudaError_t launch_combine(int dtype, const float* Y, int T, int H, int KP, void* y,
                           int num_sms, cudaStream_t st) {
  const size_t n = (size_t)T * (H / 4);
  if (n == 0) return cudaSuccess;
  size_t blocks = (n + 255) / 256;
  const size_t cap = (size_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (dtype == MOE_DTYPE_BF16)
    return launch_chained(combine_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256), 0, st,
                          1, Y, T, H, KP, (__nv_bfloat16*)y);
  return launch_chained(combine_kernel<float>, dim3((unsigned)blocks), dim3(256), 0, st, 1, Y, T,
                        H, KP, (float*)y);
}

}  // namespace moe
