// Persistent grouped GEMM over ragged expert segments on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory), fed by TMA.
//
// Problem ("GroupGEMM" section of "Lower latency and higher throughput with
// multi-node DeepSeek deployment"): g groups, group i has m_i rows, each a
// [m_i, K] x [K, N] product. Here group e < E is routed expert e with the
// positions [offsets[e], offsets[e+1]) of the permutation; group E is the
// shared expert with one row per token.
//
// Orientation: the weights are the MMA's M = 128 operand (256 on CTA pairs)
// and the tokens its N operand ("swap AB"). N is chosen per tile at run time as
// the segment's remaining rows rounded up to 16 (32 on CTA pairs, whose halves
// must each be a multiple of 16), so a ragged segment wastes at most 15 (31)
// columns, and a decode-sized segment (a handful of tokens) streams its
// expert's weights with a narrow N. The persistent tile scheduler reads the
// per-expert counts from device memory (no host round trip), as the same page
// describes for MoE under CUDA Graphs.
//
// Two products share the engine:
//  GATED (step a4, SwiGLU fused): A = 64 rows of W_gate[e] stacked over the
//    same 64 rows of W_up[e]; B = the routed token rows: for 32-token decode
//    tiles gathered from x by TMA (tile::gather4, indices from the
//    permutation, no copy of x), for larger tiles read from their
//    expert-ordered copy (the dispatch copy made by gather_rows_kernel, T*k
//    rows, unpadded). Accumulator lanes 0-63 hold gate, 64-127 up; the epilogue
//    computes silu(gate) * up and stores h rows (Qwen3.5-397B on TPU v7x,
//    4.2.1 ragged gather and 4.2.2 grouped GEMM with fused SwiGLU).
//  DOWN (step a5): A = 128 rows of W_down[e]; B = rows of h (contiguous
//    positions). The epilogue scales by the token's gate weight and stores the
//    fp32 product into the token-ordered slot buffer Y[t][r][:] (the combine
//    sums the slots afterwards in rank order).
//
// Token-operand loading (B), one of two modes:
//  kGather4 (32-token gated tiles): TMA tile::gather4, 4 rows per instruction
//    straight from x by token index (8 instructions per stage).
//  kTiled (down projection, and larger gated tiles once the routed token rows
//    were copied into expert order): the tile's rows are contiguous, one TMA
//    box per stage, the smallest of three heights that covers the tile. An SM accepts one TMA instruction only
//    every ~70-150 cycles, so a 256-token stage cannot be filled 4 rows at a
//    time; one box carries it.
// All TMA loads of a stage are issued in one SIMT step with per-lane operands.
//
// Schedule: every CTA derives the same list of units (group, feature block,
// token tile) from the offsets: the groups with rows in [m_lo, m_hi], heaviest
// first, each cut into token tiles of tile_n rows. Units are dealt round-robin
// to the persistent CTAs (or CTA pairs) through remap_unit, which interleaves
// the units of heavy groups with the light ones.
//
// CTA pairs (CL = 2, the 128- and 256-token variants): one tcgen05.mma with
// cta_group::2 spans the tensor cores of the cluster's two SMs, M = 256, N =
// the token tile. The two CTAs take adjacent feature blocks of the same group
// and token tile: each loads its own 128 weight rows (A) and one half of the
// token columns (B), so every SM stores and reads half of the token tile per
// stage instead of all of it (the shared-memory fill rate, ~90 B/clk/SM, is
// what limits a single-SM 128 x 256 tile). The leader (rank 0) waits for both
// CTAs' loads on its own full barriers, issues the MMAs, and commits their
// completion to both CTAs' empty and accumulator barriers; each CTA's epilogue
// reads its half of D from its own tensor memory and both release the
// accumulator on the leader's barrier.
//
// Warp roles: warp 0 = TMA producer, warp 1 = MMA issuer (one thread) and
// TMEM owner, warps 2-5 = epilogue (one 32-lane TMEM quarter each; the E4M3
// down GEMM has warps 2-9, two per quarter).
// A STAGES-deep shared-memory ring (full/empty mbarriers) feeds the MMA, each
// stage one or two 128-byte K boxes of both operands (NBX); two
// TMEM accumulators (tfull/tempty mbarriers) let the epilogue of one tile run
// under the main loop of the next. Every wait is bounded (status word).
#pragma once

#include <type_traits>

#include "common.cuh"

namespace moe {

struct GroupedGemmArgs {
  // GATED: [0] routed gate, [1] routed up, [2] shared gate, [3] shared up (64-row box).
  // DOWN:  [0] routed down, [2] shared down (128-row box).
  CUtensorMap tmA[4];
  // Token operand. gather4 (GATED, 32-token tiles): [0] x, 1-row box.
  // Tiled: [0..2] routed rows (expert-ordered copy of x, or h), [3..5] the
  // shared expert's rows (x, or h_shared), with boxes of B_ROWS, B_ROWS / 2
  // and 16 rows; each tile loads the smallest box that covers its columns.
  CUtensorMap tmB[6];
  const int32_t* offsets;     // [E+2]
  const int32_t* gather_idx;  // [T*k]
  const float* topk_w;        // [T*k] (DOWN)
  // E4M3 inputs only (TIn = uint8_t): power-of-two scale of every A row
  // (indexed like tmA, by the row's global index) and of every B row (GATED: x
  // rows by token, for routed and shared tiles; DOWN: [0] h rows by position,
  // [1] h_shared rows by token). Products are exact in fp32, so the epilogue
  // applies them to the accumulator without rounding.
  const float* sA[4];
  const float* sB[2];
  void* out;                  // GATED: h [T*k][I] (bf16 for E4M3 inputs); DOWN: Y fp32 [T][KP][H]
  void* out_shared;           // GATED: h_shared [T][I_shared]
  int* status;
  unsigned long long limit_ns;
  int T, k, E, KP;            // KP = k + (shared expert ? 1 : 0)
  int n_out_routed, n_out_shared;   // output features per group
  int kdim_routed, kdim_shared;     // contraction length per group
  int ld_out_routed, ld_out_shared; // row stride (elements) of out / out_shared
  unsigned flags;
  int m_lo, m_hi;             // groups with m_lo <= rows <= m_hi are scheduled
  int tile_n;                 // token tile (<= BN): a group of m rows has ceil(m / tile_n)
  // Decode-sized launches only (0 otherwise): ask L2 for the weight rows of the
  // unit each CTA is likely to take first, before waiting for the preceding
  // kernel. pf_base: raw routed A operands (GATED: gate, up; DOWN: down, unused).
  int pf_first;
  const void* pf_base[2];
  // Single-launch decode kernel only (nullptr otherwise; see fused_decode.cu).
  // GATED: unit_done[g] counts group g's finished units (h rows stored).
  // DOWN: before loading a unit's h rows, wait until unit_wait[g] holds all of
  // group g's gate/up units: ceil(rows / tile_n) * (kdim / wait_block) of them.
  int* unit_done;
  const int* unit_wait;
  int wait_block;
};

enum BMode : int { kGather4 = 0, kTiled = 2 };

template <typename TIn, bool GATED, int BN, int STAGES, int BMODE, int CL = 1, int NBX = 1>
struct GemmCfg {
  // E4M3 inputs (uint8_t codes) write bf16 h; other inputs write their own type.
  static constexpr bool F8 = sizeof(TIn) == 1;
  using TOut = std::conditional_t<F8, __nv_bfloat16, TIn>;
  static constexpr int BM = 128;                     // MMA M (weight rows)
  static constexpr int WM = GATED ? 64 : 128;        // output features per tile
  // K per stage: NBX boxes of one 128-byte row each. Two boxes give the MMA
  // issuer eight MMAs per wait and commit instead of four.
  static constexpr int BK = NBX * 128 / (int)sizeof(TIn);
  static constexpr int UMMA_K = 32 / (int)sizeof(TIn);  // K per instruction (32 bytes)
  static constexpr int A_BOX = BM * 128;                // one K box of the CTA's weight rows
  static constexpr int A_BYTES = NBX * A_BOX;
  static constexpr int B_ROWS = BN / CL;                 // token rows per CTA
  static constexpr int B_BOX = B_ROWS * 128;             // one K box of the CTA's token rows
  static constexpr int B_BYTES = NBX * B_BOX;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = (2 * BN < 32) ? 32 : 2 * BN;
  // Epilogue staging: GATED, the 128 x 32 accumulator chunk (gate and up rows
  // meet in one thread); DOWN, per-token row index and gate weight.
  static constexpr int EPI_FLOATS = GATED ? 128 * 33 + (F8 ? BN : 0) : 2 * BN;
  // Epilogue warps: 4, one per TMEM lane quarter; E4M3 DOWN, 8 (two per
  // quarter taking alternate 32-column chunks). With 1-byte operands a down
  // tile has half the k-blocks (K = I), and its stores (128 features x up to
  // 256 fp32 columns per CTA) would set the pace with one warp per quarter:
  // E4M3 prefill layer -3.4%, bf16 layers unchanged or slower by < 1%.
  static constexpr int EPI_WARPS = (!GATED && F8) ? 8 : 4;
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  static constexpr int THREADS = 64 + EPI_THREADS;
  static_assert(CL == 1 || (CL == 2 && BMODE == kTiled && BN >= 64),
                "CTA pairs split tiled token boxes of >= 64 rows");
  static_assert(NBX == 1 || (NBX == 2 && BMODE == kTiled), "two boxes per stage: tiled tokens");
  // Pair MMAs round N up to 32 (each CTA's half a multiple of 16 rows).
  static constexpr int N_ROUND = CL == 2 ? 32 : 16;
  static constexpr int KIND = UmmaOf<TIn>::kind;
  static_assert(TMEM_COLS == 32 || TMEM_COLS == 64 || TMEM_COLS == 128 || TMEM_COLS == 256 ||
                    TMEM_COLS == 512,
                "TMEM allocation must be a power of two in [32, 512]");
  static_assert(BN % 32 == 0 && BN <= 256, "token tile");

  // Heights of the three tiled token boxes (rows per CTA).
  static constexpr int BOX1 = B_ROWS / 2 < 16 ? 16 : B_ROWS / 2;

  static size_t smem_bytes(int E) {
    return 1024 /* alignment slack */ + (size_t)STAGES * STAGE_BYTES + EPI_FLOATS * 4 +
           (2 * STAGES + 5) * 8 + 16 + 3 * (size_t)(E + 2) * 4;
  }
};

struct Tile {
  int g;        // group (E = shared expert)
  int nb;       // feature block
  int mt;       // token tile inside the group
  int p0;       // first position (routed) / first token (shared)
  int n_valid;  // rows of this tile
};

// Bytes per L2 bulk prefetch instruction of the pre-wait weight prefetch.
constexpr size_t kPrefetchChunk = 32768;

// The pre-wait weight prefetch of a single-CTA GEMM (pf_first, see the pass
// below): lanes of one warp ask L2 for the WM weight rows (gate and up, or
// down) of CTA cid's likely first unit, feature block cid % nf of expert
// cid / nf. A hint only.
template <typename TIn, bool GATED, int WM>
__device__ __forceinline__ void prefetch_first_unit(const GroupedGemmArgs& args, int cid,
                                                    int lane) {
  if (!args.pf_first) return;
  const int nf = args.n_out_routed / WM;
  const int g = cid / nf;
  if (g >= args.E) return;
  const size_t row_bytes = (size_t)args.kdim_routed * sizeof(TIn);
  const size_t bytes = (size_t)WM * row_bytes;
  const size_t first = ((size_t)g * args.n_out_routed + (size_t)(cid - g * nf) * WM) * row_bytes;
  constexpr int NOP = GATED ? 2 : 1;
  const int nch = (int)((bytes + kPrefetchChunk - 1) / kPrefetchChunk);
  for (int c = lane; c < NOP * nch; c += 32) {
    const int op = c / nch;
    const size_t off = (size_t)(c - op * nch) * kPrefetchChunk;
    const size_t rem = bytes - off;
    prefetch_l2_bulk(static_cast<const uint8_t*>(args.pf_base[op]) + first + off,
                     (uint32_t)(rem < kPrefetchChunk ? rem : kPrefetchChunk));
  }
}

// Position i of the round-robin deal -> unit of the class-ordered list, whose
// first uh units belong to groups of more than 128 rows (tensor-bound tiles)
// and the rest to lighter groups (weight-streaming tiles). The heavy units are
// spread evenly over the first 7/8 of the positions (unit j at position
// floor(j * S / uh)) and the light units fill the other positions in order, so
// that SMs computing heavy tiles run beside SMs streaming light experts'
// weights, and the last positions hold short light units. A bijection.
__device__ __forceinline__ int remap_unit(int i, int total, int uh) {
  if (uh <= 0 || uh >= total) return i;
  int64_t S = (int64_t)total * 7 / 8;
  if (S < uh) S = uh;
  if (i >= S) return i;  // every heavy unit sits below S
  const int64_t j = ((int64_t)i * uh + S - 1) / S;  // heavy positions below i
  if (j < uh && j * S / uh == i) return (int)j;
  return uh + (i - (int)j);
}

// Unit u of the schedule: the scheduled groups are listed in `order` (heaviest
// first), `prefix[i]` = units of order[0..i); a group's units run feature block
// by feature block, token tile fastest, so consecutive units share weights.
__device__ __forceinline__ Tile decode_tile(int u, const int32_t* prefix, const int32_t* order,
                                            const int32_t* offs, int ngroups, int tile_n) {
  int lo = 0, hi = ngroups;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= u) lo = mid;
    else hi = mid;
  }
  Tile t;
  const int g = order[lo];
  t.g = g;
  const int m = offs[g + 1] - offs[g];
  const int mtiles = (m + tile_n - 1) / tile_n;
  const int local = u - prefix[lo];
  t.nb = local / mtiles;
  t.mt = local - t.nb * mtiles;
  t.p0 = offs[g] + t.mt * tile_n;
  t.n_valid = min(tile_n, m - t.mt * tile_n);
  return t;
}

// The unit schedule of one grouped GEMM launch, built by one warp (every CTA
// builds the same): offs <- the permutation's offsets (device-checked),
// order <- the groups with rows in [m_lo, m_hi], heaviest class first
// (> 256, > 128, > 32, the rest; group order within a class), so that the
// long tensor-bound units start first and short weight-streaming units fill
// the tail; prefix[i] <- units of order[0..i), *n_sched <- the number of
// scheduled groups, *n_heavy <- units of the groups of more than 128 rows. A
// group of m rows has ceil(m / tile_n) x (features / UNIT_FEATURES) units.
template <int UNIT_FEATURES>
__device__ __forceinline__ void build_schedule(const int32_t* offsets_src, int E, int T, int k,
                                               int KP, int m_lo, int m_hi, int tile_n,
                                               int n_out_routed, int n_out_shared, int* status,
                                               int32_t* offs, int32_t* order, int32_t* prefix,
                                               int* n_sched, int* n_heavy, int lane) {
  const int G = E + 1;
  const int tn = tile_n;
  for (int i = lane; i < G + 1; i += 32) offs[i] = offsets_src[i];
  __syncwarp();
  {
    // Device check of the permutation's offsets (once per launch): they
    // start at 0, never decrease, stay within the T*k routed positions, and
    // the shared segment holds 0 or T rows. Otherwise MOE_ERR_DEVICE_CHECK,
    // and no unit runs (every group empty), so that no tile reads or writes
    // out of its buffers.
    const int P = T * k;
    const int shared_rows = KP > k ? T : 0;
    bool bad = false;
    for (int i = lane; i < G; i += 32)
      bad |= offs[i + 1] < offs[i] || (i < E && offs[i + 1] > P);
    if (lane == 0) bad |= offs[0] != 0 || offs[E + 1] - offs[E] != shared_rows;
    if (__any_sync(0xffffffffu, bad)) {
      if (lane == 0) set_status(status, MOE_ERR_DEVICE_CHECK);
      for (int i = lane; i < G + 1; i += 32) offs[i] = 0;
      __syncwarp();
    }
  }
  auto klass = [&](int g) {
    const int m = offs[g + 1] - offs[g];
    if (m < m_lo || m > m_hi || m <= 0) return -1;
    return m > 256 ? 0 : (m > 128 ? 1 : (m > 32 ? 2 : 3));
  };
  auto units = [&](int g) {
    const int m = offs[g + 1] - offs[g];
    const int nf = (g < E ? n_out_routed : n_out_shared) / UNIT_FEATURES;
    return ((m + tn - 1) / tn) * nf;
  };
  const int per = (G + 31) / 32;
  const int g0 = lane * per, g1 = min(G, g0 + per);
  // Per-lane class counts, then a warp scan per class (registers only).
  int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
  for (int g = g0; g < g1; ++g) {
    const int c = klass(g);
    c0 += c == 0;
    c1 += c == 1;
    c2 += c == 2;
    c3 += c == 3;
  }
  auto excl_scan = [&](int v, int& total) {
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int w = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += w;
    }
    total = __shfl_sync(0xffffffffu, incl, 31);
    return incl - v;
  };
  int t0, t1, t2, t3;
  int p0 = excl_scan(c0, t0), p1 = excl_scan(c1, t1), p2 = excl_scan(c2, t2),
      p3 = excl_scan(c3, t3);
  p1 += t0;
  p2 += t0 + t1;
  p3 += t0 + t1 + t2;
  const int base = t0 + t1 + t2 + t3;
  for (int g = g0; g < g1; ++g) {
    const int c = klass(g);
    if (c == 0) order[p0++] = g;
    else if (c == 1) order[p1++] = g;
    else if (c == 2) order[p2++] = g;
    else if (c == 3) order[p3++] = g;
  }
  const int ng = base;
  __syncwarp();
  const int per2 = (ng + 31) / 32;
  const int i0 = lane * per2, i1 = min(ng, i0 + per2);
  int local = 0;
  for (int i = i0; i < i1; ++i) local += units(order[i]);
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - local;
  for (int i = i0; i < i1; ++i) {
    prefix[i] = run;
    run += units(order[i]);
  }
  if (lane == 31) {
    prefix[ng] = incl;
    *n_sched = ng;
  }
  __syncwarp();
  if (lane == 0) *n_heavy = prefix[t0 + t1];
}

// One pass of a grouped GEMM over all of its units by CTA (or CTA pair) cid of
// ncl, in the dynamic shared memory at smem_raw (GemmCfg::smem_bytes). The
// stand-alone kernel below is one pass; the single-launch decode kernel
// (fused_decode.cu) makes two, the gate/up GEMM and then the down GEMM, in the
// same shared memory: a pass leaves its mbarriers invalidated and its tensor
// memory freed. prefetch: allow the pre-wait weight prefetch (pf_first).
// FUSED (the single-launch decode kernel's passes): the permutation is read
// from offsets_in and gather_in (copies in this CTA's shared memory) instead
// of args.offsets and args.gather_idx; the gate/up pass counts its finished
// units in args.unit_done and the down pass waits on args.unit_wait; the pass
// keeps the CTA's right to allocate tensor memory unless last_alloc, and
// invalidates its mbarriers at the end. Without FUSED none of this is compiled
// in: the stand-alone kernels are the plain pass.
template <typename TIn, bool GATED, int BN, int STAGES, int BMODE, int CL, bool FUSED = false,
          int NBX = 1>
__device__ __forceinline__ void grouped_gemm_pass(const GroupedGemmArgs& args,
                                                  uint8_t* smem_raw, int cid, int ncl,
                                                  bool prefetch,
                                                  const int32_t* offsets_in = nullptr,
                                                  const int32_t* gather_in = nullptr,
                                                  bool last_alloc = true) {
  using C = GemmCfg<TIn, GATED, BN, STAGES, BMODE, CL, NBX>;
  static_assert(!FUSED || CL == 1, "the fused passes run on single CTAs");
  const int32_t* const offsets_src = FUSED ? offsets_in : args.offsets;
  const int32_t* const gather_src = FUSED ? gather_in : args.gather_idx;
  static_assert(GATED || BMODE == kTiled, "the down projection reads contiguous h rows");
  static_assert(BMODE != kGather4 || BN <= 128, "gather4 is for decode-sized token tiles");
  constexpr bool PAIR = CL == 2;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;
  float* epi = reinterpret_cast<float*>(stages + (size_t)STAGES * C::STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + C::EPI_FLOATS);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* epi_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* n_sched = reinterpret_cast<int*>(tmem_holder + 2);
  int* n_heavy = reinterpret_cast<int*>(tmem_holder + 3);  // units of groups > 128 rows
  int32_t* prefix = reinterpret_cast<int32_t*>(tmem_holder + 4);
  int32_t* offs = prefix + (args.E + 2);
  int32_t* order = offs + (args.E + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E, G = E + 1;
  // Units are walked per cluster; CTA `crank` of a pair takes feature block
  // 2 * nb + crank of each pair unit.
  const int crank = PAIR ? (int)cluster_ctarank() : 0;
  const bool leader = crank == 0;
  const uint32_t bars_base = smem_u32(bars);
  auto full_bar = [&](int s) { return bars_base + 8u * (uint32_t)s; };
  auto empty_bar = [&](int s) { return bars_base + 8u * (uint32_t)(STAGES + s); };
  auto tfull_bar = [&](int a) { return bars_base + 8u * (uint32_t)(2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bars_base + 8u * (uint32_t)(2 * STAGES + 2 + a); };
  const uint32_t stages_base = smem_u32(stages);
  const uint32_t drain_bar = smem_u32(&bars[2 * STAGES + 4]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), CL);  // a pair's leader hears both epilogues
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < 4; ++i) tma_prefetch_desc(&args.tmA[i]);
    for (int i = 0; i < 6; ++i) tma_prefetch_desc(&args.tmB[i]);
  }
  if (warp == 1) {
    if constexpr (PAIR)
      tmem_alloc_pair(smem_u32(tmem_holder), C::TMEM_COLS);
    else
      tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS, !FUSED || last_alloc);
  }
  // Weight prefetch while the preceding kernel finishes (pf_first: the host
  // sets it for decode-sized launches without a shared expert in which nearly
  // every expert holds rows, so all groups are light and scheduled in index
  // order): CTA cid's first unit would then be feature block cid % nf of
  // expert cid / nf. Until the routing is known HBM is otherwise idle; a
  // wrong guess only fetches rows that another unit reads later or that no
  // unit reads. Weights are never written by a preceding kernel, so reading
  // them before pdl_wait is safe. Not in the E4M3 gated GEMM: there the
  // layer measured 0.2-0.3% slower with it than without.
  if constexpr (!PAIR && !(GATED && C::F8)) {
    if (warp == 0 && prefetch) prefetch_first_unit<TIn, GATED, C::WM>(args, cid, lane);
  }
  pdl_wait();  // global memory from here on
  if (warp == 2)
    build_schedule<C::WM * CL>(offsets_src, args.E, args.T, args.k, args.KP, args.m_lo,
                               args.m_hi, args.tile_n, args.n_out_routed, args.n_out_shared,
                               args.status, offs, order, prefix, n_sched, n_heavy, lane);
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // peers' barriers and TMEM exist before any use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int ngroups = *n_sched;
  const int heavy_units = *n_heavy;
  const int total = prefix[ngroups];
  const uint64_t limit = args.limit_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Decode-sized tiles read each weight tile once: stream it past L2. (With
    // larger tiles evict_first measured slower: the 256-byte L2 promotion
    // fetches the next k-block's half line, which must survive until used.)
    const uint64_t pol_w = (BN <= 64) ? l2_policy_evict_first() : l2_policy_evict_normal();
    const uint64_t pol_t = l2_policy_evict_last();
    // Test hook (MOE_FLAG_TEST_SKIP_SIGNAL): the first stage of the first unit
    // is never signalled nor loaded, so the MMA issuer's wait on it runs out.
    // It is taken here, outside the k-loop: a per-k-block check in that loop
    // cost the decode step 1%.
    const bool skip_first = (args.flags & MOE_FLAG_TEST_SKIP_SIGNAL) != 0;
    uint32_t it = skip_first ? 1u : 0u;
    // Ring position of `it`, kept incrementally (the k-loop is on the decode
    // step's critical path): stage it % STAGES and phase (it / STAGES) & 1.
    int stg = (int)it;
    uint32_t ph = 0;
    int kb_first = skip_first ? 1 : 0;  // first k-block of the next unit
    bool ok = true;
    // Down GEMM of the single-launch decode kernel: the unit count of group
    // seen_g as read ahead (lane 0).
    int seen_g = -1, seen_count = 0;
    for (int u = cid; u < total && ok; u += ncl) {
      Tile tl = decode_tile(remap_unit(u, total, heavy_units), prefix, order, offs, ngroups,
                            args.tile_n);
      tl.nb = tl.nb * CL + crank;
      const bool shared = tl.g == E;
      const int kdim = shared ? args.kdim_shared : args.kdim_routed;
      if constexpr (FUSED && !GATED) {
        // Single-launch decode kernel: the group's h rows are complete once all
        // of its gate/up units have counted themselves done. The count of this
        // unit's group was read (relaxed) when the previous unit started, so
        // its L2 round trip is usually off the critical path; a value short of
        // the need is waited for with acquire loads.
        {
          int wok = 1;
          if (lane == 0) {
            const int m = offs[tl.g + 1] - offs[tl.g];
            const int need = ((m + args.tile_n - 1) / args.tile_n) * (kdim / args.wait_block);
            if (seen_g != tl.g || seen_count < need)
              wok = wait_count_at_least(args.unit_wait + tl.g, need, args.status, limit);
            fence_acq_rel_gpu();         // the relaxed read above, made an acquire
            fence_proxy_async_global();  // the TMA loads below read those h rows
            // Read ahead: the group of this CTA's next unit.
            seen_g = -1;
            if (u + ncl < total) {
              const Tile nx = decode_tile(remap_unit(u + ncl, total, heavy_units), prefix, order,
                                          offs, ngroups, args.tile_n);
              seen_g = nx.g;
              seen_count = ld_relaxed_gpu(args.unit_wait + nx.g);
            }
          }
          if (!__shfl_sync(0xffffffffu, wok, 0)) {
            ok = false;
            break;
          }
        }
      }
      const int a_row0 = (shared ? 0 : tl.g * args.n_out_routed) + tl.nb * C::WM;
      const CUtensorMap* mA0 = &args.tmA[shared ? 2 : 0];
      const CUtensorMap* mA1 = &args.tmA[shared ? 3 : 1];
      // gather4 groups: lane l issues groups q = l + 32 j (4 rows each).
      constexpr int NQ = (BMODE == kGather4) ? (BN / 4 + 31) / 32 : 1;
      int rows[NQ][4];
      int n4 = 0;
      // Tiled token box: with a pair, the MMA's N columns are split in halves;
      // the peer's half starts at column n_mma / 2 of the tile. Each CTA loads
      // the smallest of its three boxes that covers its n_mma / CL rows.
      const int n_mma = (tl.n_valid + C::N_ROUND - 1) / C::N_ROUND * C::N_ROUND;
      const int need = n_mma / CL;
      const int bsel = need <= 16 ? 2 : (need <= C::BOX1 ? 1 : 0);
      const int box_rows = bsel == 2 ? 16 : (bsel == 1 ? C::BOX1 : C::B_ROWS);
      // Bytes this stage's full barrier waits for: with a pair, the leader's
      // barrier counts both CTAs' loads.
      uint32_t tx = CL * (C::A_BYTES + NBX * box_rows * 128);
      if constexpr (BMODE == kGather4) {
        n4 = (tl.n_valid + 3) / 4;
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
          const int q = lane + 32 * j;
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int jj = min(4 * q + r, tl.n_valid - 1);
            rows[j][r] = (q < n4) ? (shared ? tl.p0 + jj - offs[E]
                                            : gather_src[tl.p0 + jj] / args.k)
                                  : 0;
          }
        }
        tx = C::A_BYTES + n4 * 4 * 128;
      }
      const int b_row0 = (shared ? tl.p0 - offs[E] : tl.p0) + crank * (n_mma / 2);
      // Per-lane operands of this tile's TMA loads (one SIMT step per stage),
      // per K box h of the stage (lanes h * PER ..): GATED: gate, up rows (+
      // token rows when tiled); DOWN: W_down rows, h rows.
      constexpr int NA = GATED ? 2 : 1;
      constexpr int PER = NA + (BMODE == kTiled ? 1 : 0);
      constexpr int NLOADS = NBX * PER;
      const int bx = lane / PER, sub = lane - bx * PER;
      const CUtensorMap* my_map = mA0;
      int my_row = a_row0;
      const int my_dx = bx * (128 / (int)sizeof(TIn));
      uint32_t my_off = (uint32_t)(bx * C::A_BOX);
      uint64_t my_pol = pol_w;
      if (GATED && sub == 1) {
        my_map = mA1;
        my_off += 64 * 128;
      }
      if (BMODE == kTiled && sub == NA) {
        my_map = &args.tmB[(shared ? 3 : 0) + bsel];
        my_row = b_row0;
        my_off = (uint32_t)(C::A_BYTES + bx * C::B_BOX);
        my_pol = pol_t;
      }
      const int nkb = kdim / C::BK;
      const int kb0 = kb_first;
      kb_first = 0;
      for (int kb = kb0; kb < nkb; ++kb) {
        const int s = stg;
        int wok = 1;
        if (lane == 0) wok = mbar_wait(empty_bar(s), ph ^ 1u, args.status, limit);
        wok = __shfl_sync(0xffffffffu, wok, 0);
        if (!wok) {
          ok = false;
          break;
        }
        ++it;
        if (++stg == STAGES) {
          stg = 0;
          ph ^= 1u;
        }
        const uint32_t a_dst = stages_base + (uint32_t)s * C::STAGE_BYTES;
        const uint32_t b_dst = a_dst + C::A_BYTES;
        const int kx = kb * C::BK;
        if constexpr (PAIR) {
          if (leader && lane == 0) mbar_arrive_expect_tx(full_bar(s), tx);
          __syncwarp();
          if (lane < NLOADS)
            tma_load_2d_pair(a_dst + my_off, my_map, kx + my_dx, my_row,
                             mapa_shared(full_bar(s), 0), my_pol);
        } else {
          if (lane == 0) mbar_arrive_expect_tx(full_bar(s), tx);
          __syncwarp();
          if (lane < NLOADS)
            tma_load_2d(a_dst + my_off, my_map, kx + my_dx, my_row, full_bar(s), my_pol);
        }
        if constexpr (BMODE == kGather4) {
#pragma unroll
          for (int j = 0; j < NQ; ++j) {
            const int q = lane + 32 * j;
            if (q < n4)
              tma_gather4(b_dst + q * 512, &args.tmB[0], kx, rows[j][0], rows[j][1], rows[j][2],
                          rows[j][3], full_bar(s), pol_t);
          }
        }
      }
    }
    // Let the last loads land before the CTA can exit (bounded, status ignored).
    // A pair's loads all complete on the leader's barriers; the leader drains
    // them, and neither CTA leaves before the closing cluster barrier.
    if (lane == 0 && leader) {
      const uint32_t n_last = it < (uint32_t)STAGES ? it : (uint32_t)STAGES;
      for (uint32_t i = it - n_last; i < it; ++i) {
        const uint32_t s = i % STAGES, round = i / STAGES;
        mbar_wait(full_bar(s), round & 1u, nullptr, 20000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      uint32_t lt = 0;
      int stg = 0;       // ring stage of the next k-block
      uint32_t ph = 0;   // its phase parity
      constexpr uint32_t fmt = UmmaOf<TIn>::fmt;
      bool ok = true;
      for (int u = cid; u < total && ok; u += ncl, ++lt) {
        Tile tl = decode_tile(remap_unit(u, total, heavy_units), prefix, order, offs, ngroups,
                            args.tile_n);
        const int kdim = (tl.g == E) ? args.kdim_shared : args.kdim_routed;
        const uint32_t acc = lt & 1u, around = lt >> 1;
        if (!mbar_wait(tempty_bar(acc), (around & 1u) ^ 1u, args.status, limit)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        const int n_mma = (tl.n_valid + C::N_ROUND - 1) / C::N_ROUND * C::N_ROUND;
        const uint32_t idesc = umma_idesc(fmt, C::BM * CL, (uint32_t)n_mma);
        for (int kb = 0; kb < kdim / C::BK; ++kb) {
          const int s = stg;
          if (!mbar_wait(full_bar(s), ph, args.status, limit)) {
            ok = false;
            break;
          }
          if (++stg == STAGES) {
            stg = 0;
            ph ^= 1u;
          }
          tc_fence_after();
          const uint32_t a_addr = stages_base + (uint32_t)s * C::STAGE_BYTES;
          const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < C::BK / C::UMMA_K; ++kk) {
            // Four MMAs per 128-byte K box.
            const uint64_t ad = umma_desc_sw128(a_addr + (kk >> 2) * C::A_BOX + (kk & 3) * 32);
            const uint64_t bd = umma_desc_sw128(b_addr + (kk >> 2) * C::B_BOX + (kk & 3) * 32);
            const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
            if constexpr (PAIR)
              umma_issue_pair<C::KIND>(d_tmem, ad, bd, idesc, accum);
            else
              umma_issue<C::KIND>(d_tmem, ad, bd, idesc, accum);
          }
          if constexpr (PAIR)
            umma_commit_pair_multicast(empty_bar(s), 0x3);
          else
            umma_commit(empty_bar(s));
        }
        if (!ok) break;
        if constexpr (PAIR)
          umma_commit_pair_multicast(tfull_bar(acc), 0x3);
        else
          umma_commit(tfull_bar(acc));
      }
      // All issued MMAs finished before TMEM is released (bounded, status ignored).
      if constexpr (PAIR)
        umma_commit_pair(drain_bar);
      else
        umma_commit(drain_bar);
      mbar_wait(drain_bar, 0, nullptr, 20000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int et = threadIdx.x - 64;        // 0..EPI_THREADS-1
    const int half = (warp - 2) >> 2;       // DOWN: which of a quarter's warps
    constexpr int NH = C::EPI_WARPS / 4;    // warps per TMEM lane quarter
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t lt = 0;
    for (int u = cid; u < total; u += ncl, ++lt) {
      Tile tl = decode_tile(remap_unit(u, total, heavy_units), prefix, order, offs, ngroups,
                            args.tile_n);
      tl.nb = tl.nb * CL + crank;
      const bool shared = tl.g == E;
      const uint32_t acc = lt & 1u, around = lt >> 1;
      if (et == 0) *epi_flag = mbar_wait(tfull_bar(acc), around & 1u, args.status, limit) ? 1 : 0;
      if constexpr (!GATED) {
        // Per-token destination row in Y and gate weight of this tile.
        int32_t* yrow = reinterpret_cast<int32_t*>(epi);
        float* wt = epi + BN;
        for (int j = et; j < tl.n_valid; j += C::EPI_THREADS) {
          int row;
          float wv;
          if (shared) {
            const int t = tl.p0 - offs[E] + j;
            row = t * args.KP + args.k;
            wv = 1.0f;
          } else {
            const int s = gather_src[tl.p0 + j];
            if ((unsigned)s < (unsigned)(args.T * args.k)) {
              const int t = s / args.k;
              row = t * args.KP + (s - t * args.k);
              wv = args.topk_w[s];
            } else {
              // Device check: a slot index out of range is reported, and its
              // column is stored as zeros into row 0 instead of out of bounds.
              set_status(args.status, MOE_ERR_DEVICE_CHECK);
              row = 0;
              wv = 0.f;
            }
          }
          // E4M3: the h row's power-of-two scale joins the gate weight (exact).
          if constexpr (C::F8) wv *= shared ? args.sB[1][tl.p0 - offs[E] + j] : args.sB[0][tl.p0 + j];
          yrow[j] = row;
          wt[j] = wv;
        }
      } else if constexpr (C::F8) {
        // Scale of each column's token row (x quantized per token).
        float* cs = epi + 128 * 33;
        for (int j = et; j < tl.n_valid; j += C::EPI_THREADS) {
          const int t = shared ? tl.p0 - offs[E] + j : gather_src[tl.p0 + j] / args.k;
          if ((unsigned)t < (unsigned)args.T) {
            cs[j] = args.sB[0][t];
          } else {  // device check, as in the down epilogue
            set_status(args.status, MOE_ERR_DEVICE_CHECK);
            cs[j] = 0.f;
          }
        }
      }
      named_barrier_sync(1, C::EPI_THREADS);
      if (!*epi_flag) break;  // every epilogue thread sees the same flag
      tc_fence_after();
      const uint32_t t_acc = tmem_base + lane_base + acc * BN;
      if constexpr (GATED) {
        using TOut = typename C::TOut;
        TOut* out = reinterpret_cast<TOut*>(shared ? args.out_shared : args.out);
        const int ld = shared ? args.ld_out_shared : args.ld_out_routed;
        const int row0 = shared ? tl.p0 - offs[E] : tl.p0;
        const int jj = et >> 2, fg = et & 3;
        // E4M3: this thread's accumulator row (lane r < 64 gate, else up row)
        // has a power-of-two scale; each column adds its token's.
        float rs = 1.0f;
        if constexpr (C::F8) {
          const int r = q * 32 + lane;
          const int f = tl.nb * 64 + (r & 63);
          const float* sa = args.sA[(shared ? 2 : 0) + (r >> 6)];
          rs = sa[(shared ? 0 : tl.g * args.n_out_routed) + f];
        }
        const float* cs = epi + 128 * 33;
        for (int c0 = 0; c0 < tl.n_valid; c0 += 32) {
          float v[32];
          tmem_ld32(t_acc + c0, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if constexpr (C::F8)
              epi[(q * 32 + lane) * 33 + i] = v[i] * (rs * cs[c0 + i]);
            else
              epi[(q * 32 + lane) * 33 + i] = v[i];
          }
          named_barrier_sync(1, C::EPI_THREADS);
          const int j = c0 + jj;
          if (j < tl.n_valid) {
            float hv[16];
#pragma unroll
            for (int f = 0; f < 16; ++f) {
              const float g = epi[(fg * 16 + f) * 33 + jj];
              const float up = epi[(64 + fg * 16 + f) * 33 + jj];
              // silu(g) * up; approximate exp and divide (a few ulp of fp32,
              // far below the bf16 rounding of h that follows).
              hv[f] = __fdividef(g, 1.0f + __expf(-g)) * up;
            }
            TOut* dst = out + (size_t)(row0 + j) * ld + tl.nb * 64 + fg * 16;
            if constexpr (sizeof(TOut) == 2) {
              uint4 pk[2];
              uint32_t* pw = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
              for (int f = 0; f < 8; ++f) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(hv[2 * f], hv[2 * f + 1]);
                pw[f] = *reinterpret_cast<const uint32_t*>(&b2);
              }
              reinterpret_cast<uint4*>(dst)[0] = pk[0];
              reinterpret_cast<uint4*>(dst)[1] = pk[1];
            } else {
#pragma unroll
              for (int f = 0; f < 4; ++f)
                reinterpret_cast<float4*>(dst)[f] =
                    make_float4(hv[4 * f], hv[4 * f + 1], hv[4 * f + 2], hv[4 * f + 3]);
            }
          }
          tc_fence_before();
          named_barrier_sync(1, C::EPI_THREADS);
        }
      } else {
        // Thread = output feature c (its TMEM lane); for each token column a
        // warp stores 32 consecutive floats of that token's slot row. The
        // epilogue warps share their schedulers with the producer and MMA
        // warps, so the per-column work is kept to one multiply and one store:
        // row indices and weights come four columns per shared-memory load.
        float* Y = reinterpret_cast<float*>(args.out);
        const int4* yrow4 = reinterpret_cast<const int4*>(epi);
        const float4* wt4 = reinterpret_cast<const float4*>(epi + BN);
        const size_t H = (size_t)args.n_out_routed;  // == n_out_shared for DOWN
        float* Yc = Y + tl.nb * 128 + q * 32 + lane;
        // E4M3: power-of-two scale of this thread's W_down row (exact).
        float rs = 1.0f;
        if constexpr (C::F8)
          rs = args.sA[shared ? 2 : 0][(shared ? 0 : (size_t)tl.g * H) + tl.nb * 128 + q * 32 +
                                       lane];
        for (int c0 = 32 * half; c0 < tl.n_valid; c0 += 32 * NH) {
          float v[32];
          tmem_ld32(t_acc + c0, v);
          if constexpr (C::F8) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= rs;
          }
          const int nj = min(32, tl.n_valid - c0);
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const int4 r = yrow4[(c0 >> 2) + i4];
            const float4 wv = wt4[(c0 >> 2) + i4];
            const int i = 4 * i4;
            if (i + 3 < nj) {
              Yc[(size_t)r.x * H] = wv.x * v[i];
              Yc[(size_t)r.y * H] = wv.y * v[i + 1];
              Yc[(size_t)r.z * H] = wv.z * v[i + 2];
              Yc[(size_t)r.w * H] = wv.w * v[i + 3];
            } else {
              if (i < nj) Yc[(size_t)r.x * H] = wv.x * v[i];
              if (i + 1 < nj) Yc[(size_t)r.y * H] = wv.y * v[i + 1];
              if (i + 2 < nj) Yc[(size_t)r.z * H] = wv.z * v[i + 2];
            }
          }
        }
        tc_fence_before();
        named_barrier_sync(1, C::EPI_THREADS);
      }
      // The accumulator goes back to the MMA issuer. Its tensor-memory reads
      // completed (tcgen05.wait::ld) before the fence and barrier above; the
      // arrive is relaxed because it orders no memory: the tile's global stores
      // are read only by later kernels (or, below, published on their own).
      if (et == 0) {
        if constexpr (PAIR)
          mbar_arrive_relaxed_cluster(mapa_shared(tempty_bar(acc), 0));
        else
          mbar_arrive_relaxed(tempty_bar(acc));
      }
      if constexpr (FUSED && GATED) {
        {
          // Single-launch decode kernel: this unit's h rows, stored by every
          // epilogue thread, become visible at GPU scope (and to the async
          // proxy that the down GEMM's TMA loads use) before the group's count
          // moves. After the accumulator's release, so that the MMA issuer
          // does not wait for these fences.
          fence_proxy_async_global();
          __threadfence();
          named_barrier_sync(1, C::EPI_THREADS);
          if (et == 0) red_release_gpu_add(args.unit_done + tl.g, 1);
        }
      }
    }
  }

  // Teardown: every MMA has completed (the leader drained them) and every
  // epilogue read of TMEM is done before either CTA of a pair frees its half.
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  if constexpr (FUSED) {
    // Every wait on the barriers has returned (the closing barrier above):
    // they can be invalidated, so that the next pass may initialise the same
    // words.
    if (threadIdx.x == 0) {
      for (int i = 0; i < 2 * STAGES + 5; ++i) mbar_inval(bars_base + 8u * (uint32_t)i);
    }
    __syncthreads();
  }
}

template <typename TIn, bool GATED, int BN, int STAGES, int BMODE, int CL, int NBX = 1>
__global__ void __launch_bounds__(GemmCfg<TIn, GATED, BN, STAGES, BMODE, CL, NBX>::THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ GroupedGemmArgs args) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  grouped_gemm_pass<TIn, GATED, BN, STAGES, BMODE, CL, false, NBX>(args, smem_raw, blockIdx.x / CL,
                                                       gridDim.x / CL, true);
}

// Host side (grouped_gemm.cu): the arguments launch_swiglu_gemm and
// launch_down_gemm pass to their kernels, for kernels that run the same passes
// (the single-launch decode kernel). False if a tensor map cannot be made.
struct GemmProblem;
struct GemmScales;
bool prepare_swiglu_gemm(GroupedGemmArgs& a, const GemmProblem& p, const void* x, const void* xg,
                         const int32_t* offsets, const int32_t* gather_idx, const void* Wg,
                         const void* Wu, const void* Wsg, const void* Wsu, void* h, void* hs,
                         int* status, const GemmScales* sc);
bool prepare_down_gemm(GroupedGemmArgs& a, const GemmProblem& p, const void* h, const void* hs,
                       const int32_t* offsets, const int32_t* gather_idx, const float* topk_w,
                       const void* Wd, const void* Wsd, float* Y, int* status,
                       const GemmScales* sc);

}  // namespace moe
