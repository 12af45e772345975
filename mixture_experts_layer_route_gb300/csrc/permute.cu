// Permutation (step a3): a stable counting sort of the routing slots by expert.
//
// "CuTeDSL at Perplexity", section "Mixture-of-Experts Dispatch/Combine",
// "Local": count the tokens routed to each expert, then give every token a
// unique index in its expert's list. The page assigns indices with atomic
// shared-memory counters (order left to the hardware); here the order is fixed
// -- ascending slot s = t*k + r inside each expert -- so that the permutation
// is reproducible and checkable bit for bit.
//
// One CTA of 32 warps. Warp w owns a contiguous chunk of slots. Pass 1 builds a
// per-warp histogram (one smem row per warp: no atomics); a column scan over
// warps and a scan over experts give each (warp, expert) its first position;
// pass 2 walks the chunk again, ranking equal experts inside each 32-slot group
// with __match_any_sync, and scatters gather_idx / slot_pos. Nothing padded is
// written: the outputs are the offsets and two index arrays.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int PM_WARPS = 32;
constexpr int PM_THREADS = PM_WARPS * 32;

__global__ void __launch_bounds__(PM_THREADS, 1)
    permute_kernel(const int32_t* __restrict__ ids, int T, int E, int k, int has_shared,
                   int32_t* __restrict__ offsets, int32_t* __restrict__ gather_idx,
                   int32_t* __restrict__ slot_pos, int* status) {
  extern __shared__ int32_t sm[];
  int32_t* hist = sm;                        // [PM_WARPS][E]
  int32_t* total = sm + PM_WARPS * E;        // [E]
  int32_t* warp_sums = total + E;            // [PM_WARPS]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = T * k;
  const int chunk = ((n + PM_WARPS * 32 - 1) / (PM_WARPS * 32)) * 32;
  const int beg = min(n, warp * chunk), end = min(n, beg + chunk);
  const uint32_t lt_mask = (1u << lane) - 1u;

  for (int i = tid; i < PM_WARPS * E; i += PM_THREADS) hist[i] = 0;
  __syncthreads();

  // Pass 1: per-warp counts.
  bool bad = false;
  for (int base = beg; base < end; base += 32) {
    const int s = base + lane;
    int e = -1;
    if (s < end) {
      e = ids[s];
      if (e < 0 || e >= E) {
        bad = true;
        e = -1;
      }
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (peers & lt_mask) == 0) hist[warp * E + e] += __popc(peers);
    __syncwarp();
  }
  if (bad) set_status(status, MOE_ERR_DEVICE_CHECK);
  __syncthreads();

  // Column scan over warps: hist[w][e] <- count of e in warps before w.
  for (int e = tid; e < E; e += PM_THREADS) {
    int run = 0;
    for (int w = 0; w < PM_WARPS; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    total[e] = run;
  }
  __syncthreads();

  // Exclusive scan of total[] over experts (E <= 1024 = one element per thread
  // per round); offsets written out.
  int carry = 0;
  for (int e0 = 0; e0 < E; e0 += PM_THREADS) {
    const int e = e0 + tid;
    const int v = (e < E) ? total[e] : 0;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int ws = warp_sums[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, ws, off);
        if (lane >= off) ws += o;
      }
      warp_sums[lane] = ws;  // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + carry;
    const int excl = before + incl - v;
    if (e < E) {
      total[e] = excl;  // now: first position of expert e
      offsets[e] = excl;
    }
    carry += warp_sums[PM_WARPS - 1];
    __syncthreads();
  }
  if (tid == 0) {
    offsets[E] = carry;
    offsets[E + 1] = carry + (has_shared ? T : 0);
  }

  // Pass 2: stable ranks and scatter.
  for (int base = beg; base < end; base += 32) {
    const int s = base + lane;
    int e = -1;
    if (s < end) {
      e = ids[s];
      if (e < 0 || e >= E) e = -1;
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int cnt = 0;
    if (e >= 0) cnt = hist[warp * E + e];
    __syncwarp();
    if (e >= 0) {
      const int p = total[e] + cnt + __popc(peers & lt_mask);
      gather_idx[p] = s;
      slot_pos[s] = p;
      if ((peers & lt_mask) == 0) hist[warp * E + e] = cnt + __popc(peers);
    } else if (s < end) {
      slot_pos[s] = -1;
    }
    __syncwarp();
  }
}

// Dispatch copy ("CuTeDSL at Perplexity", "Local": tokens are copied into
// buffers, optionally padded, for the MoE GEMM; here unpadded): row p of xg
// is x[gather_idx[p] / k], so every expert's rows are contiguous and the
// grouped GEMM reads them as one TMA box per stage. One warp per row, 16-byte
// vectors; grid sized to a multiple of the SM count.
template <int VB>
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ gather_idx,
                                                          int P, int k, int vecs_per_row,
                                                          uint4* __restrict__ xg) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int p = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < P; p += warps) {
    const int t = gather_idx[p] / k;
    const uint4* src = x + (size_t)t * vecs_per_row;
    uint4* dst = xg + (size_t)p * vecs_per_row;
    for (int v = lane; v < vecs_per_row; v += 32 * VB) {
      uint4 r[VB];
#pragma unroll
      for (int j = 0; j < VB; ++j)
        if (v + 32 * j < vecs_per_row) r[j] = __ldg(src + v + 32 * j);
#pragma unroll
      for (int j = 0; j < VB; ++j)
        if (v + 32 * j < vecs_per_row) dst[v + 32 * j] = r[j];
    }
  }
}

}  // namespace

cudaError_t launch_gather_rows(const void* x, const int32_t* gather_idx, int P, int k,
                               size_t row_bytes, void* xg, int num_sms, cudaStream_t st) {
  if (P == 0) return cudaSuccess;
  const int vpr = (int)(row_bytes / 16);
  int blocks = (P + 7) / 8;
  if (blocks > 8 * num_sms) blocks = 8 * num_sms;
  gather_rows_kernel<4><<<blocks, 256, 0, st>>>(reinterpret_cast<const uint4*>(x), gather_idx, P,
                                                k, vpr, reinterpret_cast<uint4*>(xg));
  return cudaGetLastError();
}

size_t permute_smem_bytes(int E) { return sizeof(int32_t) * ((size_t)PM_WARPS * E + E + PM_WARPS); }

cudaError_t launch_permute(const int32_t* ids, int T, int E, int k, int has_shared,
                           int32_t* offsets, int32_t* gather_idx, int32_t* slot_pos, int* status,
                           cudaStream_t st) {
  const size_t smem = permute_smem_bytes(E);
  cudaError_t err = cudaFuncSetAttribute(permute_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  permute_kernel<<<1, PM_THREADS, smem, st>>>(ids, T, E, k, has_shared, offsets, gather_idx,
                                              slot_pos, status);
  return cudaGetLastError();
}

}  // namespace moe
