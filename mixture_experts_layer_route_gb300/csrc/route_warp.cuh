// Top-k routing of one token by one warp (step a2), shared by the route kernel
// (router.cu) and the single-launch decode kernel (fused_decode.cu).
#pragma once

#include "common.cuh"

namespace moe {

// Order-preserving key of a float: for non-NaN a, b, a > b exactly when
// key(a) > key(b). -0 is taken as +0 first, so the two zeros tie as they do
// under float comparison. key_value inverts it (returning +0 for either zero).
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

constexpr uint32_t kNoExpert = 0xffffffffu;

// Arg-max over the warp: the largest key among the lanes' candidates (bi !=
// kNoExpert), and among equal keys the lowest index. Two warp reductions.
__device__ __forceinline__ uint32_t warp_argmax(uint32_t bk, uint32_t bi, uint32_t* best_key) {
  const uint32_t mx = __reduce_max_sync(0xffffffffu, bi == kNoExpert ? 0u : bk);
  *best_key = mx;
  return __reduce_min_sync(0xffffffffu, (bi != kNoExpert && bk == mx) ? bi : kNoExpert);
}

// Top-k and gate weights of one token by one warp. v[i] holds the logit of
// expert lane + 32 i. k rounds of warp arg-max over the experts not yet
// chosen, ties to the lower expert index; lane r keeps round r. Values are
// compared as order-preserving integer keys, so a round is a lane-local scan
// and two warp reductions.
// Group-limited form (n_group > 1, the DeepSeek router of the same section, of
// which plain top-k is the one-group case): the experts form n_group
// contiguous groups of E / n_group; a group's score is its largest logit; only
// the topk_group best groups (lower group index among equals) take part in the
// k rounds. Gate weights use the unmasked logits.
template <int NV>
__device__ __forceinline__ void route_warp(const float (&v)[NV], int E, int k, int renorm,
                                           int n_group, int topk_group,
                                           int32_t* __restrict__ ids_row,
                                           float* __restrict__ w_row) {
  const int lane = threadIdx.x & 31;
  uint32_t key[NV];
  uint32_t live = 0;  // bit i: expert lane + 32 i exists and can still be chosen
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    key[i] = order_key(v[i]);
    if (lane + 32 * i < E) live |= 1u << i;
  }
  if (n_group > 1) {
    const int G = E / n_group;
    int grp[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) grp[i] = (lane + 32 * i) / G;  // >= n_group past E
    uint32_t gkey = 0;  // lane j < n_group: key of group j's largest logit
    for (int j = 0; j < n_group; ++j) {
      uint32_t mk = 0;
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (grp[i] == j) mk = max(mk, key[i]);
      mk = __reduce_max_sync(0xffffffffu, mk);
      if (lane == j) gkey = mk;
    }
    uint32_t kept = 0;
    for (int r = 0; r < topk_group; ++r) {
      const bool cand = lane < n_group && !((kept >> lane) & 1u);
      uint32_t unused;
      const uint32_t g = warp_argmax(gkey, cand ? (uint32_t)lane : kNoExpert, &unused);
      if (g < 32u) kept |= 1u << g;
    }
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (grp[i] >= n_group || !((kept >> grp[i]) & 1u)) live &= ~(1u << i);
  }
  uint32_t my_key = 0;
  int my_idx = 0;
  for (int r = 0; r < k; ++r) {
    uint32_t bk = 0, bi = kNoExpert;
#pragma unroll
    for (int i = 0; i < NV; ++i) {  // ascending expert index: the first maximum wins
      if (((live >> i) & 1u) && (bi == kNoExpert || key[i] > bk)) {
        bk = key[i];
        bi = (uint32_t)(lane + 32 * i);
      }
    }
    uint32_t mx;
    const uint32_t win = warp_argmax(bk, bi, &mx);
    if (win != kNoExpert && (int)(win & 31u) == lane) live &= ~(1u << (win >> 5));
    if (lane == r) {
      my_key = mx;
      my_idx = (int)win;
    }
  }

  const float m = key_value(__shfl_sync(0xffffffffu, my_key, 0));
  const float p = (lane < k) ? expf(key_value(my_key) - m) : 0.f;
  float ssum;
  if (renorm) {
    ssum = p;
  } else {
    ssum = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (lane + 32 * i < E) ssum += expf(key_value(key[i]) - m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, off);
  if (lane < k) {
    ids_row[lane] = my_idx;
    w_row[lane] = p / ssum;
  }
}

}  // namespace moe
