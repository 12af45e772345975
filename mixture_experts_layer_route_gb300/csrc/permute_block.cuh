// Block-level stable counting sort of the routing slots by expert, shared by
// the stand-alone permutation kernels (32 warps) and the single-launch decode
// kernel (6 warps, fused_decode.cu). See permute.cu for the method.
#pragma once

#include "common.cuh"

namespace moe {

// sm: NW * E + E + NW ints of shared memory. CG: read the ids through L2 only
// (they were written by other CTAs of the same launch).
template <int NW, bool CG>
__device__ __forceinline__ void permute_block(const int32_t* __restrict__ ids, int T, int E,
                                              int k, int has_shared,
                                              int32_t* __restrict__ offsets,
                                              int32_t* __restrict__ gather_idx,
                                              int32_t* __restrict__ slot_pos, int* status,
                                              int32_t* sm) {
  constexpr int PM_WARPS = NW, PM_THREADS = NW * 32;
  int32_t* hist = sm;                        // [NW][E]
  int32_t* total = sm + NW * E;              // [E]
  int32_t* warp_sums = total + E;            // [NW]
  auto load_id = [&](int s) { return CG ? __ldcg(ids + s) : ids[s]; };

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
      e = load_id(s);
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
      int ws = lane < NW ? warp_sums[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, ws, off);
        if (lane >= off) ws += o;
      }
      if (lane < NW) warp_sums[lane] = ws;  // inclusive over warps
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
      e = load_id(s);
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

}  // namespace moe
