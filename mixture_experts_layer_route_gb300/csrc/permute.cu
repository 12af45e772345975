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
#include "permute_block.cuh"

namespace moe {

namespace {

constexpr int PM_WARPS = 32;
constexpr int PM_THREADS = PM_WARPS * 32;

__global__ void __launch_bounds__(PM_THREADS, 1)
    permute_kernel(const int32_t* __restrict__ ids, int T, int E, int k, int has_shared,
                   int32_t* __restrict__ offsets, int32_t* __restrict__ gather_idx,
                   int32_t* __restrict__ slot_pos, int* status) {
  pdl_entry();
  extern __shared__ int32_t sm[];
  permute_block<PM_WARPS, false>(ids, T, E, k, has_shared, offsets, gather_idx, slot_pos, status,
                                 sm);
}

// Large T*k: the same stable order from two grid-wide kernels. Chunk c owns
// slots [c*CHUNK, (c+1)*CHUNK). The first kernel writes each chunk's expert
// counts to chunk_hist[c][e]; the second recomputes, per CTA, the global
// offsets (a scan over experts of the column sums) and its chunk's base
// (offsets + counts of the earlier chunks), then ranks and scatters its slots
// exactly like the single-CTA kernel.
constexpr int PM_CHUNK = 2048;

__global__ void __launch_bounds__(PM_THREADS, 1)
    permute_count_kernel(const int32_t* __restrict__ ids, int n, int E,
                         int32_t* __restrict__ chunk_hist, int* status) {
  pdl_entry();
  extern __shared__ int32_t sm[];
  int32_t* hist = sm;  // [E]
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int e = tid; e < E; e += PM_THREADS) hist[e] = 0;
  __syncthreads();
  const int beg = blockIdx.x * PM_CHUNK, end = min(n, beg + PM_CHUNK);
  bool bad = false;
  for (int base = beg + (tid & ~31); base < end; base += PM_THREADS) {
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
    if (e >= 0 && (peers & lt_mask) == 0) atomicAdd(&hist[e], __popc(peers));
  }
  if (bad) set_status(status, MOE_ERR_DEVICE_CHECK);
  __syncthreads();
  for (int e = tid; e < E; e += PM_THREADS) chunk_hist[(size_t)blockIdx.x * E + e] = hist[e];
}

__global__ void __launch_bounds__(PM_THREADS, 1)
    permute_scatter_kernel(const int32_t* __restrict__ ids, int T, int E, int k, int has_shared,
                           const int32_t* __restrict__ chunk_hist, int32_t* __restrict__ offsets,
                           int32_t* __restrict__ gather_idx, int32_t* __restrict__ slot_pos) {
  pdl_entry();
  extern __shared__ int32_t sm[];
  int32_t* hist = sm;                        // [PM_WARPS][E]
  int32_t* total = sm + PM_WARPS * E;        // [E]: chunk base of expert e
  int32_t* warp_sums = total + E;            // [PM_WARPS]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = T * k;
  const int c = blockIdx.x, nchunk = gridDim.x;
  const int cbeg = c * PM_CHUNK, cend = min(n, cbeg + PM_CHUNK);
  const int per = PM_CHUNK / PM_WARPS;  // 64 slots per warp
  const int beg = min(cend, cbeg + warp * per), end = min(cend, beg + per);
  const uint32_t lt_mask = (1u << lane) - 1u;

  // Column sums over chunks (all of them, and those before this chunk).
  for (int e = tid; e < E; e += PM_THREADS) {
    int all = 0, before = 0;
    for (int cc = 0; cc < nchunk; ++cc) {
      const int v = chunk_hist[(size_t)cc * E + e];
      if (cc < c) before += v;
      all += v;
    }
    total[e] = all;
    hist[e] = before;  // parked in warp 0's row until the scan is done
  }
  for (int i = tid; i < PM_WARPS * E; i += PM_THREADS)
    if (i >= E) hist[i] = 0;
  __syncthreads();

  // Exclusive scan of the expert totals -> offsets; chunk base = offset + before.
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
      warp_sums[lane] = ws;
    }
    __syncthreads();
    const int excl = (warp > 0 ? warp_sums[warp - 1] : 0) + carry + incl - v;
    if (e < E) {
      if (c == 0) offsets[e] = excl;
      total[e] = excl + hist[e];
    }
    carry += warp_sums[PM_WARPS - 1];
    __syncthreads();
  }
  if (c == 0 && tid == 0) {
    offsets[E] = carry;
    offsets[E + 1] = carry + (has_shared ? T : 0);
  }
  for (int e = tid; e < E; e += PM_THREADS) hist[e] = 0;
  __syncthreads();

  // Per-warp counts inside this chunk, then a column scan over warps.
  for (int b = beg; b < end; b += 32) {
    const int s = b + lane;
    int e = -1;
    if (s < end) {
      e = ids[s];
      if (e < 0 || e >= E) e = -1;
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (peers & lt_mask) == 0) hist[warp * E + e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = tid; e < E; e += PM_THREADS) {
    int run = 0;
    for (int w = 0; w < PM_WARPS; ++w) {
      const int cnt = hist[w * E + e];
      hist[w * E + e] = run;
      run += cnt;
    }
  }
  __syncthreads();

  // Stable ranks and scatter.
  for (int b = beg; b < end; b += 32) {
    const int s = b + lane;
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
// buffers, optionally padded, for the MoE GEMM; here unpadded): row
// slot_pos[s] of xg is x[s / k], so every expert's rows are contiguous and the
// grouped GEMM reads them as one TMA box per stage. One warp per slot, in slot
// order: the k warps that copy one token's row run together and read it from
// L2 (x is read from DRAM once), while each writes a whole row. (In position
// order, the 8x larger stream of written rows evicted x from L2 between
// re-reads: 0.136 against 0.097 ms for the 8192-token prefill batch.) Slots
// with slot_pos < 0 (out-of-range ids) have no row; a position beyond the T*k
// rows is a device-check failure (MOE_ERR_DEVICE_CHECK) and is not copied.
// 16-byte vectors, 4 KB per warp in flight; streaming stores.
template <int VB>
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ slot_pos,
                                                          int P, int k, int vecs_per_row,
                                                          uint4* __restrict__ xg, int* status) {
  pdl_entry();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int s = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; s < P; s += warps) {
    const int p = slot_pos[s];
    if (p < 0) continue;
    if (p >= P) {
      if (lane == 0) set_status(status, MOE_ERR_DEVICE_CHECK);
      continue;
    }
    const uint4* src = x + (size_t)(s / k) * vecs_per_row;
    uint4* dst = xg + (size_t)p * vecs_per_row;
    for (int v = lane; v < vecs_per_row; v += 32 * VB) {
      uint4 r[VB];
#pragma unroll
      for (int j = 0; j < VB; ++j)
        if (v + 32 * j < vecs_per_row) r[j] = __ldg(src + v + 32 * j);
#pragma unroll
      for (int j = 0; j < VB; ++j)
        if (v + 32 * j < vecs_per_row) __stcs(dst + v + 32 * j, r[j]);
    }
  }
}

}  // namespace

cudaError_t launch_gather_rows(const void* x, const int32_t* slot_pos, int P, int k,
                               size_t row_bytes, void* xg, int* status, int num_sms,
                               cudaStream_t st) {
  if (P == 0) return cudaSuccess;
  const int vpr = (int)(row_bytes / 16);
  int blocks = (P + 7) / 8;
  if (blocks > 16 * num_sms) blocks = 16 * num_sms;
  return launch_chained(gather_rows_kernel<8>, dim3(blocks), dim3(256), 0, st, 1,
                        reinterpret_cast<const uint4*>(x), slot_pos, P, k, vpr,
                        reinterpret_cast<uint4*>(xg), status);
}

size_t permute_smem_bytes(int E) { return sizeof(int32_t) * ((size_t)PM_WARPS * E + E + PM_WARPS); }

// Up to this many slots one CTA does the whole permutation; above it, chunks.
constexpr int64_t kPermuteSingleMax = 4096;

int64_t permute_chunks(int64_t T, int64_t k) {
  const int64_t n = T * k;
  return n <= kPermuteSingleMax ? 0 : (n + PM_CHUNK - 1) / PM_CHUNK;
}

size_t permute_scratch_bytes(int64_t T, int64_t E, int64_t k) {
  return (size_t)permute_chunks(T, k) * (size_t)E * sizeof(int32_t);
}

cudaError_t launch_permute(const int32_t* ids, int T, int E, int k, int has_shared,
                           int32_t* offsets, int32_t* gather_idx, int32_t* slot_pos, int* status,
                           int32_t* chunk_hist, cudaStream_t st) {
  const size_t smem = permute_smem_bytes(E);
  const int nchunk = (int)permute_chunks(T, k);
  cudaError_t err;
  if (nchunk == 0) {
    err = cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (err != cudaSuccess) return err;
    return launch_chained(permute_kernel, dim3(1), dim3(PM_THREADS), smem, st, 1, ids, T, E, k,
                          has_shared, offsets, gather_idx, slot_pos, status);
  }
  err = cudaFuncSetAttribute(permute_scatter_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  err = launch_chained(permute_count_kernel, dim3(nchunk), dim3(PM_THREADS),
                       (size_t)E * sizeof(int32_t), st, 1, ids, T * k, E, chunk_hist, status);
  if (err != cudaSuccess) return err;
  return launch_chained(permute_scatter_kernel, dim3(nchunk), dim3(PM_THREADS), smem, st, 1, ids,
                        T, E, k, has_shared, (const int32_t*)chunk_hist, offsets, gather_idx,
                        slot_pos);
}

}  // namespace moe
