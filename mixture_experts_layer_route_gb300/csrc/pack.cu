// Weight packing: a row-major [rows][cols] matrix into tiles of 64 rows x 128
// bytes, tile (rb, kb) contiguous at ((rb * nkb + kb) * 8 KB), nkb = row bytes
// / 128. The grouped GEMMs then read one 64-row k-step of a weight tile as a
// single 8 KB block. A pure byte permutation: one thread per 16-byte vector,
// reads and writes coalesced within each 128-byte piece.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

__global__ void __launch_bounds__(256)
    pack_tiles_kernel(const uint4* __restrict__ src, int64_t rows, int64_t nkb,
                      uint4* __restrict__ dst) {
  const int64_t n = rows * nkb * 8;  // 16-byte vectors
  for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < n;
       v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tile = v >> 9;     // 512 vectors per 8 KB tile
    const int within = (int)(v & 511);
    const int r = within >> 3, c = within & 7;
    const int64_t rb = tile / nkb, kb = tile - rb * nkb;
    dst[v] = src[(rb * 64 + r) * (nkb * 8) + kb * 8 + c];
  }
}

}  // namespace

cudaError_t launch_pack_tiles(const void* src, int64_t rows, int64_t row_bytes, void* dst,
                              int num_sms, cudaStream_t st) {
  const int64_t nkb = row_bytes / 128;
  const int64_t n = rows * nkb * 8;
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
  pack_tiles_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<const uint4*>(src), rows,
                                                      nkb, reinterpret_cast<uint4*>(dst));
  return cudaGetLastError();
}

}  // namespace moe
