// moe_down_combine_noalloc: the down projection + combine for callers that
// cannot allocate device memory.
//
// Some callers own no device allocator: a host application that hands the
// layer only its input and output buffers, a plugin whose host forbids
// cudaMalloc at run time, or code under a fixed device-memory budget. They
// cannot provide the workspace moe_down_combine needs (the fp32 slot buffer and
// the status word). This entry point runs the same kernels with that scratch
// in one file-scope device array instead, so it needs no workspace argument
// and allocates nothing.
//
// The array is a static __device__ object of this library: every GPU that
// loads the library holds it until the process exits. Its address is taken
// once per device with cudaGetSymbolAddress (host code must not use the
// array's name as a device pointer: on the host it is only a stand-in).
#include <mutex>

#include "moe_api.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// 256-byte header (the status word) followed by the fp32 slot buffer.
constexpr size_t kNoAllocHeader = 256;
constexpr size_t kNoAllocSlotBytes = (size_t)16 << 20;  // 16 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocHeader + kNoAllocSlotBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the array on the current device, looked up on the first
// call made with that device current.
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_down_combine_noalloc(const moe_problem* pb, const void* h,
                                               const void* h_shared,
                                               const int32_t* expert_offsets,
                                               const int32_t* gather_idx, const float* topk_w,
                                               const void* W_down, const void* Ws_down, void* y,
                                               void* stream, moe_status* device_status) {
  // The same checks as moe_down_combine, int32 index ranges included.
  moe_status s = check_problem(pb);
  if (s != MOE_OK) return s;
  const moe_problem& p = *pb;
  if (p.T == 0) return MOE_OK;
  const bool has_s = p.I_shared > 0;
  if (!h || !expert_offsets || !gather_idx || !topk_w || !W_down || !y) return MOE_ERR_INVALID_ARG;
  if (has_s != (Ws_down != nullptr) || has_s != (h_shared != nullptr)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {h, expert_offsets, gather_idx, topk_w, W_down, y};
  for (const void* q : ptrs)
    if (!is_aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (has_s && (!is_aligned16(Ws_down) || !is_aligned16(h_shared))) return MOE_ERR_INVALID_ARG;
  // The slot buffer holds T x (k + shared) rows of H fp32 values.
  const size_t KP = (size_t)p.k + (has_s ? 1 : 0);
  const size_t slot_bytes = (size_t)p.T * KP * (size_t)p.H * 4;
  if (slot_bytes > kNoAllocSlotBytes) return MOE_ERR_WORKSPACE;
  if (!tensor_map_encoder_available()) return MOE_ERR_UNSUPPORTED;

  void* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  int* status = reinterpret_cast<int*>(scratch);
  float* Y = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(scratch) + kNoAllocHeader);

  const GemmProblem g = gemm_problem(p);
  cudaStream_t st = (cudaStream_t)stream;
  // The status word must start each call at MOE_OK; the slot rows are all
  // overwritten by the down-projection epilogue before the combine reads them.
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), st);
  if (e == cudaSuccess)
    e = launch_down_gemm(g, h, h_shared, expert_offsets, gather_idx, topk_w, W_down, Ws_down, Y,
                         status, st);
  if (e == cudaSuccess)
    e = launch_combine(p.out_f32 ? MOE_DTYPE_F32 : p.dtype, Y, g.T, g.H, (int)KP, y, g.num_sms,
                       st);
  if (e == cudaSuccess && device_status) {
    int v = 0;
    e = cudaMemcpyAsync(&v, status, sizeof(int), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) *device_status = (moe_status)v;
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
