// Grouped GEMMs of the MXFP8 layer: expert weights stored as E4M3 codes with
// one E8M0 scale per block of 32 elements along the contraction axis
// ("Hosting Qwen on Blackwell", quantization section: MXFP8 weights converted
// statically; "CuTeDSL at Perplexity", Blackwell quantization paragraph: the
// absolute maximum over 32 elements), token operands as bf16 rows holding
// MXFP8 values (x quantized per forward pass, h quantized in the gate/up
// epilogue).
//
// The weights stream from HBM as codes (1 byte per element plus 1/32 for the
// scales) and are turned into their exact bf16 values on the SM, so the
// product runs on the bf16 tensor-core MMA (kind::f16): a code times a power
// of two is a bf16 value (exactly, for scales of 2^-117 and up), and the MMA
// sums exact products in fp32, which is the block-scaled product up to the
// order of the fp32 sums.
//
// Problem and schedule as grouped_gemm.cuh (the same unit list and deal); the
// differences are in the pipeline of one CTA (no CTA pairs). Two tile shapes,
// chosen per problem: when the experts average 256 routed rows or more,
// 256-token tiles with K = 64 per stage (each converted weight tile serves
// twice the tokens); otherwise 128-token tiles with K = 128 per stage.
//   warp 0, token producer: per stage the token tile (boxes of BN tokens x
//     64 bf16 elements) into a ring of STAGES stages.
//   warp 10, code producer: per stage the 128 weight rows' codes (one BK-byte
//     box per 64 or 128 rows; 64-byte swizzle for K = 64, 128-byte for K =
//     128) into a ring of CST stages of its own, and per unit the scale panel
//     of its weight rows (all K / 32 scale bytes of each row, one box per 64
//     or 128 rows) into one of two panel buffers. The codes run ahead of the
//     token tiles, so their conversion is off the loop a token stage goes
//     through (MMA done -> refill -> MMA).
//   warps 6-9, converters (one per TMEM lane quarter, thread = weight row):
//     once a stage's codes landed and the slot of its token stage is free
//     (the MMAs of that stage's previous round completed), the row's codes
//     times their block scales -> bf16 pairs, stored into the slot (the MMA
//     reads operand A from there: row m in lane m, column c holding elements
//     2c and 2c + 1), then one arrive per warp on the stage's "converted"
//     barrier and on the code stage's "empty" one.
//   warp 1, MMA issuer: per stage a wait for the token tile and one for the
//     converted slot, BK / 16 MMAs of K = 16 (A from the slot, B from the
//     token stage, K-major, 128-byte swizzle) into the accumulator (two of 128
//     columns, or one of 256 beside the slots), and one commit that frees the
//     token stage and its slot together.
//   warps 2-5, epilogue: GATED, silu(gate) * up, then each h row quantized per
//     block of 32 features (the two threads holding a block's 16 + 16 values
//     share their maximum) and stored as its bf16 values; DOWN, as the bf16
//     layer: gate weight applied, fp32 slot rows.
// Every wait is bounded (status word).
#include "grouped_gemm.cuh"
#include "kernels.h"
#include "mx.cuh"

namespace moe {

struct MxGemmArgs {
  // E4M3 weight codes, rows of K bytes. GATED: [0] routed gate, [1] routed up,
  // [2] shared gate, [3] shared up (64-row boxes); DOWN: [0] routed down, [2]
  // shared down (128-row boxes). Boxes of BK bytes: 64 (64-byte swizzle) or
  // 128 (128-byte swizzle).
  CUtensorMap tmA[4];
  // The E8M0 scale rows of the same weights (sk bytes per row), indexed like
  // tmA; a box holds whole rows (sk bytes) of 64 or 128 rows, no swizzle.
  CUtensorMap tmS[4];
  // bf16 token rows, tiled: [0..2] routed rows by position (the expert-ordered
  // copy of x, or h), [3..5] the shared expert's rows by token (x, or
  // h_shared); boxes of BN, BN / 2 (at least 16) and 16 rows.
  CUtensorMap tmB[6];
  const int32_t* offsets;     // [E+2]
  const int32_t* gather_idx;  // [T*k] (DOWN)
  const float* topk_w;        // [T*k] (DOWN)
  void* out;                  // GATED: h bf16 [T*k][I]; DOWN: Y fp32 [T][KP][H]
  void* out_shared;           // GATED: h_shared bf16 [T][I_shared]
  int* status;
  unsigned long long limit_ns;
  int T, k, E, KP;
  int n_out_routed, n_out_shared;   // output features per group
  int kdim_routed, kdim_shared;     // contraction length per group
  int sk_routed, sk_shared;         // scale bytes per weight row
  int ld_out_routed, ld_out_shared;
  unsigned flags;
  int m_lo, m_hi, tile_n;
  // Decode kernel only (mx_dec_kernel; unused by mx_gemm_kernel): tmB then
  // holds E4M3 token codes (128-byte boxes, 128-byte swizzle) and tmSB their
  // scale rows, whole rows of 32 tokens: [0] routed rows by position, [1] the
  // shared expert's by token.
  CUtensorMap tmSB[2];
  int skb_routed, skb_shared;       // scale bytes per token row of the B operand
  // GATED: scale rows of h / h_shared (the MXFP8 codes go to out / out_shared).
  uint8_t* out_scales;
  uint8_t* out_shared_scales;
  int sko_routed, sko_shared;       // their bytes per row
};

namespace {

template <bool GATED, int BN, int STAGES, int CST, int BK_>
struct MxCfg {
  static constexpr int BM = 128;                 // weight rows per unit (MMA M)
  static constexpr int WM = GATED ? 64 : 128;    // output features per unit
  static constexpr int BK = BK_;                 // K per stage: 128 or 64
  static constexpr int A8_BYTES = BM * BK;       // codes of one stage (BK-byte rows)
  static constexpr int NBH = BK / 64;            // token boxes per stage (64 bf16 elements each)
  static constexpr int B_HALF = BN * 128;
  static constexpr int STAGE_BYTES = NBH * B_HALF;  // token ring stage (STAGES of them)
  // A converted stage in tensor memory: one slot per shared-memory stage, so
  // a slot is free again exactly when its stage is (the same MMAs read both).
  static constexpr int SLOT_COLS = BK / 2;
  // Two fp32 accumulators when they fit beside the converted slots, else one
  // (256-token tiles: the epilogue then overlaps only the next unit's loads
  // and conversion, not its MMAs).
  static constexpr int NACC = 2 * BN + STAGES * SLOT_COLS <= 512 ? 2 : 1;
  static constexpr int ACC_COLS = NACC * BN;
  static constexpr int TMEM_COLS = 512;
  static constexpr int EPI_FLOATS = GATED ? 128 * 33 : 2 * BN;
  // token producer, MMA, 4 epilogue, 4 converter warps, code producer
  static constexpr int THREADS = 352;
  static constexpr int BOX1 = BN / 2 < 16 ? 16 : BN / 2;
  // full, empty, cfull [STAGES]; afull, aempty [CST]; pfull, pempty, tfull, tempty [2]; drain
  static constexpr int NBARS = 3 * STAGES + 2 * CST + 9;
  static_assert(ACC_COLS + STAGES * SLOT_COLS <= TMEM_COLS, "tensor memory");
  static_assert(BK == 64 || BK == 128, "stage depth");
  static_assert(BN % 32 == 0 && BN <= 256, "token tile");
  static_assert(STAGE_BYTES % 1024 == 0 && A8_BYTES % 1024 == 0, "stage alignment");

  static size_t smem_bytes(int E, int sk_max) {
    return 1024 + (size_t)STAGES * STAGE_BYTES + (size_t)CST * A8_BYTES +
           2 * (size_t)BM * sk_max + EPI_FLOATS * 4 + NBARS * 8 + 16 + 3 * (size_t)(E + 2) * 4;
  }
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// tcgen05.mma kind::f16 with operand A in tensor memory (address a_tmem).
__device__ __forceinline__ void umma_issue_tmem_a(uint32_t d_tmem, uint32_t a_tmem,
                                                  uint64_t bdesc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Each thread of the warp writes 32 consecutive 32-bit columns of its own
// TMEM lane (the warp's lane quarter is in taddr's lane field).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Each thread reads 64 consecutive fp32 columns of its own TMEM lane (the
// warp's lane quarter is in taddr's lane field); the wait is in the same
// statement, so no use of the registers precedes it.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, "
      "%45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, "
      "%62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]),
        "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
        "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]),
        "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// (a0, a1) += (p0 * s0, p1 * s1) * sa with packed fp32 pair instructions (one
// multiply and one fused multiply-add for the two lanes of the pair; each
// element is rounded exactly as fmaf(p * s, sa, a)).
__device__ __forceinline__ void mul_fma2(float& a0, float& a1, float p0, float p1, float s0,
                                         float s1, float sa) {
  asm("{\n\t.reg .b64 pp, ps, pt, pa, pc;\n\t"
      "mov.b64 pp, {%2, %3};\n\t"
      "mov.b64 ps, {%4, %5};\n\t"
      "mul.rn.f32x2 pt, pp, ps;\n\t"
      "mov.b64 pa, {%6, %6};\n\t"
      "mov.b64 pc, {%0, %1};\n\t"
      "fma.rn.f32x2 pc, pt, pa, pc;\n\t"
      "mov.b64 {%0, %1}, pc;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(p0), "f"(p1), "f"(s0), "f"(s1), "f"(sa));
}

// acc[n] += P_b[n] * s_B[n][b] * s_A[b] over this warp's two blocks b = 2 bh,
// 2 bh + 1 and the tile's NC columns (P: the two partials, NC columns each;
// fkb: the stage's token scales as floats, [4 blocks][32]; sw: the weight
// row's four scale bytes of the stage).
template <int NC>
__device__ __forceinline__ void scale_blocks(const float (&P)[2 * NC], float (&acc)[32],
                                             uint32_t sw, int bh, const float* fkb) {
#pragma unroll
  for (int bb = 0; bb < 2; ++bb) {
    const int b = 2 * bh + bb;
    const float sa = mx_scale_of((sw >> (8 * b)) & 0xFFu);
    const float4* fb = reinterpret_cast<const float4*>(fkb + b * 32);
#pragma unroll
    for (int n4 = 0; n4 < NC / 4; ++n4) {
      const float4 sb = fb[n4];
      mul_fma2(acc[4 * n4 + 0], acc[4 * n4 + 1], P[bb * NC + 4 * n4 + 0], P[bb * NC + 4 * n4 + 1],
               sb.x, sb.y, sa);
      mul_fma2(acc[4 * n4 + 2], acc[4 * n4 + 3], P[bb * NC + 4 * n4 + 2], P[bb * NC + 4 * n4 + 3],
               sb.z, sb.w, sa);
    }
  }
}

// All lanes wait (each thread's own acquire of the phase); the warp agrees on
// the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* status,
                                          uint64_t limit) {
  const bool ok = mbar_wait(bar, parity, status, limit);
  return __all_sync(0xffffffffu, ok);
}

template <bool GATED, int BN, int STAGES, int CST, int BK>
__global__ void __launch_bounds__(MxCfg<GATED, BN, STAGES, CST, BK>::THREADS, 1)
    mx_gemm_kernel(const __grid_constant__ MxGemmArgs args) {
  pdl_trigger();
  using C = MxCfg<GATED, BN, STAGES, CST, BK>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int E = args.E;
  const int sk_max = args.sk_routed > args.sk_shared ? args.sk_routed : args.sk_shared;
  const int panel_bytes = C::BM * sk_max;
  uint8_t* stages = smem;                                       // token ring
  uint8_t* astages = stages + (size_t)STAGES * C::STAGE_BYTES;  // code ring
  uint8_t* panels = astages + (size_t)CST * C::A8_BYTES;
  float* epi = reinterpret_cast<float*>(panels + 2 * (size_t)panel_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + C::EPI_FLOATS);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::NBARS);
  volatile int* epi_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* n_sched = reinterpret_cast<int*>(tmem_holder + 2);
  int* n_heavy = reinterpret_cast<int*>(tmem_holder + 3);
  int32_t* prefix = reinterpret_cast<int32_t*>(tmem_holder + 4);
  int32_t* offs = prefix + (E + 2);
  int32_t* order = offs + (E + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bars_base = smem_u32(bars);
  auto full_bar = [&](int s) { return bars_base + 8u * (uint32_t)s; };
  auto empty_bar = [&](int s) { return bars_base + 8u * (uint32_t)(STAGES + s); };
  auto cfull_bar = [&](int s) { return bars_base + 8u * (uint32_t)(2 * STAGES + s); };
  auto afull_bar = [&](int j) { return bars_base + 8u * (uint32_t)(3 * STAGES + j); };
  auto aempty_bar = [&](int j) { return bars_base + 8u * (uint32_t)(3 * STAGES + CST + j); };
  constexpr int B0 = 3 * STAGES + 2 * CST;
  auto pfull_bar = [&](int p) { return bars_base + 8u * (uint32_t)(B0 + p); };
  auto pempty_bar = [&](int p) { return bars_base + 8u * (uint32_t)(B0 + 2 + p); };
  auto tfull_bar = [&](int a) { return bars_base + 8u * (uint32_t)(B0 + 4 + a); };
  auto tempty_bar = [&](int a) { return bars_base + 8u * (uint32_t)(B0 + 6 + a); };
  const uint32_t drain_bar = bars_base + 8u * (uint32_t)(B0 + 8);
  const uint32_t stages_base = smem_u32(stages);
  const uint32_t astages_base = smem_u32(astages);
  const uint32_t panels_base = smem_u32(panels);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(cfull_bar(s), 4);  // one arrive per converter warp
    }
    for (int j = 0; j < CST; ++j) {
      mbar_init(afull_bar(j), 1);
      mbar_init(aempty_bar(j), 4);  // one arrive per converter warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(pfull_bar(i), 1);
      mbar_init(pempty_bar(i), 4);
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), 1);
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < 4; ++i) tma_prefetch_desc(&args.tmA[i]);
    for (int i = 0; i < 4; ++i) tma_prefetch_desc(&args.tmS[i]);
    for (int i = 0; i < 6; ++i) tma_prefetch_desc(&args.tmB[i]);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
  pdl_wait();  // global memory from here on
  if (warp == 2)
    build_schedule<C::WM>(args.offsets, E, args.T, args.k, args.KP, args.m_lo, args.m_hi,
                          args.tile_n, args.n_out_routed, args.n_out_shared, args.status, offs,
                          order, prefix, n_sched, n_heavy, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int ngroups = *n_sched;
  const int heavy_units = *n_heavy;
  const int total = prefix[ngroups];
  const uint64_t limit = args.limit_ns;
  const int cid = blockIdx.x, ncl = gridDim.x;
  auto tile_of = [&](int u) {
    return decode_tile(remap_unit(u, total, heavy_units), prefix, order, offs, ngroups,
                       args.tile_n);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ token producer
    const uint64_t pol_t = l2_policy_evict_last();
    // Test hook (MOE_FLAG_TEST_SKIP_SIGNAL): the first token stage is never
    // loaded, so the MMA issuer's wait on it runs out.
    const bool skip_first = (args.flags & MOE_FLAG_TEST_SKIP_SIGNAL) != 0;
    uint32_t it = skip_first ? 1u : 0u;
    int stg = (int)it;
    uint32_t ph = 0;
    int kb_first = skip_first ? 1 : 0;
    bool ok = true;
    for (int u = cid; u < total && ok; u += ncl) {
      const Tile tl = tile_of(u);
      const bool shared = tl.g == E;
      const int kdim = shared ? args.kdim_shared : args.kdim_routed;
      const int n_mma = (tl.n_valid + 15) / 16 * 16;
      const int bsel = n_mma <= 16 ? 2 : (n_mma <= C::BOX1 ? 1 : 0);
      const int box_rows = bsel == 2 ? 16 : (bsel == 1 ? C::BOX1 : BN);
      const uint32_t tx = (uint32_t)(C::NBH * box_rows * 128);
      const int b_row0 = shared ? tl.p0 - offs[E] : tl.p0;
      const CUtensorMap* my_map = &args.tmB[(shared ? 3 : 0) + bsel];
      const int nkb = kdim / C::BK;
      const int kb0 = kb_first;
      kb_first = 0;
      for (int kb = kb0; kb < nkb; ++kb) {
        const int s = stg;
        int wok = 1;
        if (lane == 0) wok = mbar_wait(empty_bar(s), ph ^ 1u, args.status, limit);
        if (!__shfl_sync(0xffffffffu, wok, 0)) {
          ok = false;
          break;
        }
        ++it;
        if (++stg == STAGES) {
          stg = 0;
          ph ^= 1u;
        }
        const uint32_t dst = stages_base + (uint32_t)s * C::STAGE_BYTES;
        if (lane == 0) mbar_arrive_expect_tx(full_bar(s), tx);
        __syncwarp();
        // Lane h: the tile's h-th box of 64 bf16 elements.
        if (lane < C::NBH)
          tma_load_2d(dst + (uint32_t)(lane * C::B_HALF), my_map, kb * C::BK + 64 * lane, b_row0,
                      full_bar(s), pol_t);
      }
    }
    // Let the last loads land before the CTA can exit (bounded, status ignored).
    if (lane == 0) {
      const uint32_t n_last = it < (uint32_t)STAGES ? it : (uint32_t)STAGES;
      for (uint32_t i = it - n_last; i < it; ++i)
        mbar_wait(full_bar((int)(i % STAGES)), (i / STAGES) & 1u, nullptr, 20000000ull);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ------------------------------------------------------------ code producer
    // Weight codes run ahead of the token tiles in their own ring, so their
    // conversion is done before the MMA needs the slot.
    const uint64_t pol_w = BN <= 64 ? l2_policy_evict_first() : l2_policy_evict_normal();
    uint32_t it = 0, aph = 0;
    int ast = 0;
    bool ok = true;
    uint32_t lt = 0;
    constexpr int NA = GATED ? 2 : 1;
    for (int u = cid; u < total && ok; u += ncl, ++lt) {
      const Tile tl = tile_of(u);
      const bool shared = tl.g == E;
      const int kdim = shared ? args.kdim_shared : args.kdim_routed;
      const int sk = shared ? args.sk_shared : args.sk_routed;
      const int a_row0 = (shared ? 0 : tl.g * args.n_out_routed) + tl.nb * C::WM;
      // The unit's scale panel.
      {
        const int p = (int)(lt & 1u);
        int wok = 1;
        if (lane == 0) wok = mbar_wait(pempty_bar(p), ((lt >> 1) & 1u) ^ 1u, args.status, limit);
        if (!__shfl_sync(0xffffffffu, wok, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(pfull_bar(p), (uint32_t)(C::BM * sk));
        __syncwarp();
        const uint32_t pdst = panels_base + (uint32_t)(p * panel_bytes);
        if (lane < NA)
          tma_load_2d(pdst + (uint32_t)(lane * 64 * sk), &args.tmS[(shared ? 2 : 0) + lane], 0,
                      a_row0, pfull_bar(p), pol_w);
      }
      // Lanes < NA: the weight codes (GATED: gate, up rows; one BK-byte box of
      // 64 or 128 rows each).
      const CUtensorMap* my_map = &args.tmA[(shared ? 2 : 0) + (GATED && lane == 1 ? 1 : 0)];
      const uint32_t my_off = GATED && lane == 1 ? 64u * C::BK : 0u;
      const int nkb = kdim / C::BK;
      for (int kb = 0; kb < nkb; ++kb) {
        const int j = ast;
        int wok = 1;
        if (lane == 0) wok = mbar_wait(aempty_bar(j), aph ^ 1u, args.status, limit);
        if (!__shfl_sync(0xffffffffu, wok, 0)) {
          ok = false;
          break;
        }
        ++it;
        if (++ast == CST) {
          ast = 0;
          aph ^= 1u;
        }
        const uint32_t dst = astages_base + (uint32_t)j * C::A8_BYTES;
        if (lane == 0) mbar_arrive_expect_tx(afull_bar(j), (uint32_t)C::A8_BYTES);
        __syncwarp();
        if (lane < NA) tma_load_2d(dst + my_off, my_map, kb * C::BK, a_row0, afull_bar(j), pol_w);
      }
    }
    // Let the last loads land before the CTA can exit (bounded, status ignored).
    if (lane == 0) {
      const uint32_t n_last = it < (uint32_t)CST ? it : (uint32_t)CST;
      for (uint32_t i = it - n_last; i < it; ++i)
        mbar_wait(afull_bar((int)(i % CST)), (i / CST) & 1u, nullptr, 20000000ull);
      const uint32_t p_last = lt < 2u ? lt : 2u;
      for (uint32_t i = lt - p_last; i < lt; ++i)
        mbar_wait(pfull_bar((int)(i & 1u)), (i >> 1) & 1u, nullptr, 20000000ull);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t lt = 0, ph = 0;
      int stg = 0;
      bool ok = true;
      for (int u = cid; u < total && ok; u += ncl, ++lt) {
        const Tile tl = tile_of(u);
        const int kdim = (tl.g == E) ? args.kdim_shared : args.kdim_routed;
        const uint32_t acc = lt % C::NACC, around = lt / C::NACC;
        if (!mbar_wait(tempty_bar((int)acc), (around & 1u) ^ 1u, args.status, limit)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        const int n_mma = (tl.n_valid + 15) / 16 * 16;
        const uint32_t idesc = umma_idesc(1, C::BM, (uint32_t)n_mma);
        for (int kb = 0; kb < kdim / C::BK; ++kb) {
          // The stage's token tile and its converted weight slot.
          const int s = stg;
          if (!mbar_wait(full_bar(s), ph, args.status, limit) ||
              !mbar_wait(cfull_bar(s), ph, args.status, limit)) {
            ok = false;
            break;
          }
          if (++stg == STAGES) {
            stg = 0;
            ph ^= 1u;
          }
          tc_fence_after();
          const uint32_t a_t = tmem_base + C::ACC_COLS + (uint32_t)(s * C::SLOT_COLS);
          const uint32_t b_addr = stages_base + (uint32_t)s * C::STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk)
            umma_issue_tmem_a(d_tmem, a_t + (uint32_t)kk * 8u,
                              umma_desc_sw128(b_addr + (kk >> 2) * C::B_HALF + (kk & 3) * 32),
                              idesc, (kb | kk) != 0 ? 1u : 0u);
          // Frees the token stage and its slot together (the converters wait
          // on the same barrier before writing the slot again).
          umma_commit(empty_bar(s));
        }
        if (!ok) break;
        umma_commit(tfull_bar((int)acc));
      }
      umma_commit(drain_bar);
      mbar_wait(drain_bar, 0, nullptr, 20000000ull);
    }
    __syncwarp();
  } else if (warp >= 6 && warp < 10) {
    // ------------------------------------------------------------ converters
    const int q = warp & 3;
    const int r = q * 32 + lane;  // weight row of the unit = TMEM lane
    const uint32_t lane_field = (uint32_t)(q * 32) << 16;
    uint32_t lt = 0, ph = 0, aph = 0;
    int stg = 0, ast = 0;
    bool ok = true;
    for (int u = cid; u < total && ok; u += ncl, ++lt) {
      const Tile tl = tile_of(u);
      const bool shared = tl.g == E;
      const int kdim = shared ? args.kdim_shared : args.kdim_routed;
      const int sk = shared ? args.sk_shared : args.sk_routed;
      const int p = (int)(lt & 1u);
      if (!warp_wait(pfull_bar(p), (lt >> 1) & 1u, args.status, limit)) break;
      const uint8_t* srow = panels + (size_t)p * panel_bytes + (size_t)r * sk;
      for (int kb = 0; kb < kdim / C::BK; ++kb) {
        // The codes of this k-block, and the slot of its token stage free:
        // the MMAs of that stage's previous round completed (no later round
        // can complete before this warp's arrival on cfull).
        const int s = stg, j = ast;
        if (!warp_wait(afull_bar(j), aph, args.status, limit) ||
            !warp_wait(empty_bar(s), ph ^ 1u, args.status, limit)) {
          ok = false;
          break;
        }
        if (++stg == STAGES) {
          stg = 0;
          ph ^= 1u;
        }
        if (++ast == CST) {
          ast = 0;
          aph ^= 1u;
        }
        tc_fence_after();
        // BK / 32 scale bytes per stage (blocks BK / 32 * kb ..).
        const uint32_t sw = C::BK == 128 ? *reinterpret_cast<const uint32_t*>(srow + kb * 4)
                                         : *reinterpret_cast<const uint16_t*>(srow + kb * 2);
        // BK-byte rows: 128-byte swizzle (chunk j of row r at j ^ (r & 7)) or
        // 64-byte swizzle (at j ^ ((r >> 1) & 3)).
        const uint8_t* arow = astages + (size_t)j * C::A8_BYTES + (size_t)r * C::BK;
        const int rsw = C::BK == 128 ? (r & 7) : ((r >> 1) & 3);
#pragma unroll
        for (int h = 0; h < C::NBH; ++h) {
          uint32_t o[32];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = 4 * h + jj;  // 16-byte chunk of the row
            const uint4 ch = *reinterpret_cast<const uint4*>(arow + ((j ^ rsw) << 4));
            const float X = mx_scale_of((sw >> (8 * (j >> 1))) & 0xFFu);
            mx_decode4_bf16(ch.x, X, o[8 * jj + 0], o[8 * jj + 1]);
            mx_decode4_bf16(ch.y, X, o[8 * jj + 2], o[8 * jj + 3]);
            mx_decode4_bf16(ch.z, X, o[8 * jj + 4], o[8 * jj + 5]);
            mx_decode4_bf16(ch.w, X, o[8 * jj + 6], o[8 * jj + 7]);
          }
          tmem_st32(tmem_base + lane_field + C::ACC_COLS + (uint32_t)(s * C::SLOT_COLS + h * 32),
                    o);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(cfull_bar(s));
          mbar_arrive(aempty_bar(j));
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(pempty_bar(p));
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int et = threadIdx.x - 64;  // 0..127
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t lt = 0;
    for (int u = cid; u < total; u += ncl, ++lt) {
      Tile tl = tile_of(u);
      const bool shared = tl.g == E;
      const uint32_t acc = lt % C::NACC, around = lt / C::NACC;
      if (et == 0)
        *epi_flag = mbar_wait(tfull_bar((int)acc), around & 1u, args.status, limit) ? 1 : 0;
      if constexpr (!GATED) {
        int32_t* yrow = reinterpret_cast<int32_t*>(epi);
        float* wt = epi + BN;
        for (int j = et; j < tl.n_valid; j += 128) {
          int row;
          float wv;
          if (shared) {
            const int t = tl.p0 - offs[E] + j;
            row = t * args.KP + args.k;
            wv = 1.0f;
          } else {
            const int s = args.gather_idx[tl.p0 + j];
            if ((unsigned)s < (unsigned)(args.T * args.k)) {
              const int t = s / args.k;
              row = t * args.KP + (s - t * args.k);
              wv = args.topk_w[s];
            } else {  // device check: reported; the column goes to row 0 as zeros
              set_status(args.status, MOE_ERR_DEVICE_CHECK);
              row = 0;
              wv = 0.f;
            }
          }
          yrow[j] = row;
          wt[j] = wv;
        }
      }
      named_barrier_sync(1, 128);
      if (!*epi_flag) break;
      tc_fence_after();
      const uint32_t t_acc = tmem_base + lane_base + acc * BN;
      if constexpr (GATED) {
        __nv_bfloat16* out =
            reinterpret_cast<__nv_bfloat16*>(shared ? args.out_shared : args.out);
        const int ld = shared ? args.ld_out_shared : args.ld_out_routed;
        const int row0 = shared ? tl.p0 - offs[E] : tl.p0;
        const int jj = et >> 2, fg = et & 3;
        for (int c0 = 0; c0 < tl.n_valid; c0 += 32) {
          float v[32];
          tmem_ld32(t_acc + c0, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) epi[(q * 32 + lane) * 33 + i] = v[i];
          named_barrier_sync(1, 128);
          float hv[16];
          float amax = 0.0f;
#pragma unroll
          for (int f = 0; f < 16; ++f) {
            const float g = epi[(fg * 16 + f) * 33 + jj];
            const float up = epi[(64 + fg * 16 + f) * 33 + jj];
            hv[f] = __fdividef(g, 1.0f + __expf(-g)) * up;
            amax = fmaxf(amax, fabsf(hv[f]));
          }
          // Block of 32 features: this thread's 16 and its neighbour's (fg ^ 1).
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          const int e = mx_block_exponent(amax);
          const float inv = mx_pow2(-e), X = mx_pow2(e);
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            mx_decode4_bf16(mx_encode4(hv[4 * i] * inv, hv[4 * i + 1] * inv,
                                       hv[4 * i + 2] * inv, hv[4 * i + 3] * inv),
                            X, pk[2 * i], pk[2 * i + 1]);
          const int j = c0 + jj;
          if (j < tl.n_valid) {
            uint4* dst = reinterpret_cast<uint4*>(out + (size_t)(row0 + j) * ld + tl.nb * 64 +
                                                  fg * 16);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
          tc_fence_before();
          named_barrier_sync(1, 128);
        }
      } else {
        float* Y = reinterpret_cast<float*>(args.out);
        const int4* yrow4 = reinterpret_cast<const int4*>(epi);
        const float4* wt4 = reinterpret_cast<const float4*>(epi + BN);
        const size_t H = (size_t)args.n_out_routed;
        float* Yc = Y + tl.nb * 128 + q * 32 + lane;
        for (int c0 = 0; c0 < tl.n_valid; c0 += 32) {
          float v[32];
          tmem_ld32(t_acc + c0, v);
          const int nj = min(32, tl.n_valid - c0);
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const int4 rr = yrow4[(c0 >> 2) + i4];
            const float4 wv = wt4[(c0 >> 2) + i4];
            const int i = 4 * i4;
            if (i < nj) Yc[(size_t)rr.x * H] = wv.x * v[i];
            if (i + 1 < nj) Yc[(size_t)rr.y * H] = wv.y * v[i + 1];
            if (i + 2 < nj) Yc[(size_t)rr.z * H] = wv.z * v[i + 2];
            if (i + 3 < nj) Yc[(size_t)rr.w * H] = wv.w * v[i + 3];
          }
        }
        tc_fence_before();
        named_barrier_sync(1, 128);
      }
      if (et == 0) mbar_arrive_relaxed(tempty_bar((int)acc));
    }
  }

  // Teardown: every MMA has completed (drained), every tensor-memory access of
  // the epilogue and the converters is done.
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Decode-sized MXFP8 GEMMs (32-token tiles): E4M3 x E4M3 on the tensor cores
// (kind::f8f6f4), with the block scales applied by the CUDA cores. The MMA's
// K = 32 is exactly one MXFP8 block, so every MMA writes one block's partial
// product P_b (fp32, exact sums of exact code products) into its own slot of
// tensor memory; scaler warps read the partials and accumulate
//   acc[m][n] += P_b[m][n] * s_B[n][b] * s_A[m][b]
// in registers (both scales are powers of two: the products are exact and the
// one rounding per block is the fp32 accumulation, as in the MMA itself). At
// decode sizes an MMA's time is set by its A bytes, so E4M3 operands run twice
// as fast as their bf16 values would.
//
// Warp roles: warp 0 producer (per stage: the weight codes and the token
// codes; per unit: the scale rows of the unit's weight rows and of its token
// tile, into one of two panel buffers), warp 1 MMA issuer (four MMAs per stage into one of four
// slot groups of tensor memory), warps 2-9 scalers and epilogue (warp w: TMEM
// lane quarter w % 4, blocks 2 bh and 2 bh + 1 of every stage for
// bh = (w - 2) / 4, all token columns; the two halves' sums are added in
// shared memory).
// GATED epilogue: silu(gate) * up, quantized per 32 features (MXFP8 codes and
// scale bytes of h); DOWN: the gate-weighted fp32 slot rows, as mx_gemm_kernel.

template <bool GATED, int STAGES>
struct MxDecCfg {
  static constexpr int BN = 32;
  static constexpr int BM = 128;
  static constexpr int WM = GATED ? 64 : 128;
  static constexpr int BK = 128;
  static constexpr int A_BYTES = BM * 128;   // codes
  static constexpr int B_BYTES = BN * 128;   // token codes
  static constexpr int B_OFF = A_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 20 KB
  static constexpr int NG = 4;               // partial slot groups (4 blocks x 32 columns)
  static constexpr int TMEM_COLS = 512;
  static constexpr int SCALER_WARPS = 8;
  static constexpr int THREADS = 64 + 32 * SCALER_WARPS;
  // Partial sums of the two scaler halves meet here (128 rows x 32 columns,
  // padded), then DOWN's per-column destination rows and gate weights. The
  // space is shared with the token scales as floats (fpanel), which are dead
  // by then.
  static constexpr int EPI_FLOATS = 128 * 33 + 2 * BN;
  // full, empty [STAGES]; pfull, pempty [NG]; scale panels full, empty [2]; drain
  static constexpr int NBARS = 2 * STAGES + 2 * NG + 5;
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(NG * 4 * BN <= TMEM_COLS, "tensor memory");

  // skb_max: scale bytes per row of the weights and of the tokens (the same
  // contraction axis); nblk_max: 32-element blocks of K.
  static size_t smem_bytes(int E, int skb_max, int nblk_max) {
    const size_t fp = (size_t)nblk_max * BN;
    return 1024 + (size_t)STAGES * STAGE_BYTES + 2 * (size_t)(BM + BN) * skb_max +
           4 * (fp > (size_t)EPI_FLOATS ? fp : (size_t)EPI_FLOATS) + NBARS * 8 + 16 +
           3 * (size_t)(E + 2) * 4;
  }
};

template <bool GATED, int STAGES>
__global__ void __launch_bounds__(MxDecCfg<GATED, STAGES>::THREADS, 1)
    mx_dec_kernel(const __grid_constant__ MxGemmArgs args) {
  pdl_trigger();
  using C = MxDecCfg<GATED, STAGES>;
  constexpr int BN = C::BN;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int E = args.E;
  const int skb_max = args.skb_routed > args.skb_shared ? args.skb_routed : args.skb_shared;
  const int kmax = args.kdim_routed > args.kdim_shared ? args.kdim_routed : args.kdim_shared;
  const int nblk_max = kmax / 32;
  // Per unit, in one of two panel buffers: the weight rows' scale rows
  // [BM][skb] followed by the token tile's [BN][skb].
  const int panel_bytes = (C::BM + BN) * skb_max;
  uint8_t* stages = smem;
  uint8_t* panels = stages + (size_t)STAGES * C::STAGE_BYTES;
  float* fpanel = reinterpret_cast<float*>(panels + 2 * (size_t)panel_bytes);  // [blk][BN]
  float* epi = fpanel;  // used only after the unit's last stage
  const size_t fp_floats = (size_t)nblk_max * BN;
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      fpanel + (fp_floats > (size_t)C::EPI_FLOATS ? fp_floats : (size_t)C::EPI_FLOATS));
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* n_sched = reinterpret_cast<int*>(tmem_holder + 2);
  int* n_heavy = reinterpret_cast<int*>(tmem_holder + 3);
  int32_t* prefix = reinterpret_cast<int32_t*>(tmem_holder + 4);
  int32_t* offs = prefix + (E + 2);
  int32_t* order = offs + (E + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bars_base = smem_u32(bars);
  auto full_bar = [&](int s) { return bars_base + 8u * (uint32_t)s; };
  auto empty_bar = [&](int s) { return bars_base + 8u * (uint32_t)(STAGES + s); };
  auto pfull_bar = [&](int g) { return bars_base + 8u * (uint32_t)(2 * STAGES + g); };
  auto pempty_bar = [&](int g) { return bars_base + 8u * (uint32_t)(2 * STAGES + C::NG + g); };
  constexpr int B0 = 2 * STAGES + 2 * C::NG;
  auto bfull_bar = [&](int p) { return bars_base + 8u * (uint32_t)(B0 + p); };
  auto bempty_bar = [&](int p) { return bars_base + 8u * (uint32_t)(B0 + 2 + p); };
  const uint32_t drain_bar = bars_base + 8u * (uint32_t)(B0 + 4);
  const uint32_t stages_base = smem_u32(stages);
  const uint32_t panels_base = smem_u32(panels);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int g = 0; g < C::NG; ++g) {
      mbar_init(pfull_bar(g), 1);
      mbar_init(pempty_bar(g), C::SCALER_WARPS);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bfull_bar(i), 1);
      mbar_init(bempty_bar(i), C::SCALER_WARPS);
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
    *abort_flag = 0;
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < 4; ++i) tma_prefetch_desc(&args.tmA[i]);
    for (int i = 0; i < 4; ++i) tma_prefetch_desc(&args.tmS[i]);
    for (int i = 0; i < 6; ++i) tma_prefetch_desc(&args.tmB[i]);
    for (int i = 0; i < 2; ++i) tma_prefetch_desc(&args.tmSB[i]);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
  pdl_wait();  // global memory from here on
  if (warp == 2)
    build_schedule<C::WM>(args.offsets, E, args.T, args.k, args.KP, args.m_lo, args.m_hi,
                          args.tile_n, args.n_out_routed, args.n_out_shared, args.status, offs,
                          order, prefix, n_sched, n_heavy, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int ngroups = *n_sched;
  const int heavy_units = *n_heavy;
  const int total = prefix[ngroups];
  const uint64_t limit = args.limit_ns;
  const int cid = blockIdx.x, ncl = gridDim.x;
  auto tile_of = [&](int u) {
    return decode_tile(remap_unit(u, total, heavy_units), prefix, order, offs, ngroups,
                       args.tile_n);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_t = l2_policy_evict_last();
    const bool skip_first = (args.flags & MOE_FLAG_TEST_SKIP_SIGNAL) != 0;
    uint32_t it = skip_first ? 1u : 0u;
    int stg = (int)it;
    uint32_t ph = 0;
    int kb_first = skip_first ? 1 : 0;
    bool ok = true;
    uint32_t lt = 0;
    constexpr int NA = GATED ? 2 : 1;
    constexpr int NLOADS = NA + 1;  // weight codes, token codes
    for (int u = cid; u < total && ok; u += ncl, ++lt) {
      const Tile tl = tile_of(u);
      const bool shared = tl.g == E;
      const int kdim = shared ? args.kdim_shared : args.kdim_routed;
      const int skb = shared ? args.skb_shared : args.skb_routed;
      const int a_row0 = (shared ? 0 : tl.g * args.n_out_routed) + tl.nb * C::WM;
      const int b_row0 = shared ? tl.p0 - offs[E] : tl.p0;
      {  // the unit's scale panels: weight rows (one box per 64 / 128 rows), token rows
        const int p = (int)(lt & 1u);
        int wok = 1;
        if (lane == 0) wok = mbar_wait(bempty_bar(p), ((lt >> 1) & 1u) ^ 1u, args.status, limit);
        if (!__shfl_sync(0xffffffffu, wok, 0)) {
          ok = false;
          break;
        }
        const uint32_t pdst = panels_base + (uint32_t)(p * panel_bytes);
        if (lane == 0) mbar_arrive_expect_tx(bfull_bar(p), (uint32_t)((C::BM + BN) * skb));
        __syncwarp();
        if (lane < NA)
          tma_load_2d(pdst + (uint32_t)(lane * 64 * skb), &args.tmS[(shared ? 2 : 0) + lane], 0,
                      a_row0, bfull_bar(p), pol_w);
        else if (lane == NA)
          tma_load_2d(pdst + (uint32_t)(C::BM * skb), &args.tmSB[shared ? 1 : 0], 0, b_row0,
                      bfull_bar(p), pol_t);
      }
      const int n_mma = (tl.n_valid + 15) / 16 * 16;
      const int bsel = n_mma <= 16 ? 2 : 0;
      const int box_rows = n_mma <= 16 ? 16 : BN;
      const uint32_t tx = C::A_BYTES + (uint32_t)box_rows * 128u;
      // Per-lane operands: lanes < NA weight codes (GATED: gate, up rows),
      // lane NA the token codes.
      const CUtensorMap* my_map = &args.tmA[(shared ? 2 : 0) + (lane % NA)];
      int my_row = a_row0;
      uint32_t my_off = (uint32_t)((lane % NA) * 64 * 128);
      uint64_t my_pol = pol_w;
      if (lane == NA) {
        my_map = &args.tmB[(shared ? 3 : 0) + bsel];
        my_row = b_row0;
        my_off = C::B_OFF;
        my_pol = pol_t;
      }
      const int nkb = kdim / C::BK;
      const int kb0 = kb_first;
      kb_first = 0;
      for (int kb = kb0; kb < nkb; ++kb) {
        const int s = stg;
        int wok = 1;
        if (lane == 0) wok = mbar_wait(empty_bar(s), ph ^ 1u, args.status, limit);
        if (!__shfl_sync(0xffffffffu, wok, 0)) {
          ok = false;
          break;
        }
        ++it;
        if (++stg == STAGES) {
          stg = 0;
          ph ^= 1u;
        }
        const uint32_t dst = stages_base + (uint32_t)s * C::STAGE_BYTES;
        if (lane == 0) mbar_arrive_expect_tx(full_bar(s), tx);
        __syncwarp();
        if (lane < NLOADS) tma_load_2d(dst + my_off, my_map, kb * C::BK, my_row, full_bar(s), my_pol);
      }
    }
    if (lane == 0) {
      const uint32_t n_last = it < (uint32_t)STAGES ? it : (uint32_t)STAGES;
      for (uint32_t i = it - n_last; i < it; ++i)
        mbar_wait(full_bar((int)(i % STAGES)), (i / STAGES) & 1u, nullptr, 20000000ull);
      const uint32_t p_last = lt < 2u ? lt : 2u;
      for (uint32_t i = lt - p_last; i < lt; ++i)
        mbar_wait(bfull_bar((int)(i & 1u)), (i >> 1) & 1u, nullptr, 20000000ull);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t i = 0;  // global stage index
      bool ok = true;
      for (int u = cid; u < total && ok; u += ncl) {
        const Tile tl = tile_of(u);
        const int kdim = (tl.g == E) ? args.kdim_shared : args.kdim_routed;
        const int n_mma = (tl.n_valid + 15) / 16 * 16;
        const uint32_t idesc = umma_idesc(UmmaOf<uint8_t>::fmt, C::BM, (uint32_t)n_mma);
        // Partial slot of block b in group g: column g * 4 BN + b * n_mma (a
        // 16-column tile packs its four partials into half of the group).
        for (int kb = 0; kb < kdim / C::BK; ++kb, ++i) {
          const int s = (int)(i % STAGES), g = (int)(i % C::NG);
          if (!mbar_wait(full_bar(s), (i / STAGES) & 1u, args.status, limit) ||
              !mbar_wait(pempty_bar(g), ((i / C::NG) & 1u) ^ 1u, args.status, limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = stages_base + (uint32_t)s * C::STAGE_BYTES;
          const uint32_t b_addr = a_addr + C::B_OFF;
#pragma unroll
          for (int b = 0; b < 4; ++b)
            umma_issue<kKindF8>(tmem_base + (uint32_t)(g * 4 * BN + b * n_mma),
                                umma_desc_sw128(a_addr + b * 32), umma_desc_sw128(b_addr + b * 32),
                                idesc, 0u);
          umma_commit(empty_bar(s));
          umma_commit(pfull_bar(g));
        }
      }
      umma_commit(drain_bar);
      mbar_wait(drain_bar, 0, nullptr, 20000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ scalers + epilogue
    // Warp w: TMEM lane quarter w % 4 (thread = weight row), blocks 2 bh and
    // 2 bh + 1 of every stage (bh = (w - 2) / 4), all token columns; the two
    // halves' sums are added in shared memory. Every decision to stop is taken
    // from the shared abort flag after a barrier, so that all scaler warps
    // pass the same barriers.
    const int q = warp & 3;
    const int bh = (warp - 2) >> 2;
    const int r = q * 32 + lane;  // weight row of the unit = TMEM lane
    const int et = threadIdx.x - 64;  // 0..255
    constexpr int NT = 32 * C::SCALER_WARPS;
    const uint32_t t_quarter = tmem_base + ((uint32_t)(q * 32) << 16);
    uint32_t lt = 0, i = 0;
    for (int u = cid; u < total; u += ncl, ++lt) {
      const Tile tl = tile_of(u);
      const bool shared = tl.g == E;
      const int kdim = shared ? args.kdim_shared : args.kdim_routed;
      const int skb = shared ? args.skb_shared : args.skb_routed;
      const int nblk = kdim / 32;
      // Token scales of the tile as floats, block-major: fpanel[b][n].
      const int p = (int)(lt & 1u);
      if (et == 0 && !mbar_wait(bfull_bar(p), (lt >> 1) & 1u, args.status, limit))
        *abort_flag = 1;
      named_barrier_sync(1, NT);
      if (*abort_flag) break;
      mbar_wait(bfull_bar(p), (lt >> 1) & 1u, nullptr, limit);  // completed: this thread's acquire
      const uint8_t* apanel = panels + (size_t)p * panel_bytes;  // [BM][skb]
      {
        const uint8_t* bp = apanel + (size_t)C::BM * skb;       // [BN][skb]
        for (int e = et; e < nblk * BN; e += NT) {
          const int b = e / BN, n = e - b * BN;
          fpanel[e] = mx_scale_of(bp[n * skb + b]);
        }
      }
      named_barrier_sync(1, NT);
      const uint8_t* srow = apanel + (size_t)r * skb;
      uint4 sc4 = make_uint4(0, 0, 0, 0);
      // Tiles of at most 16 tokens (the usual decode tile) have 16-column
      // partials: half the tensor-memory reads and multiply-adds.
      const bool n16 = tl.n_valid <= 16;
      const uint32_t t_lane = t_quarter + (uint32_t)(bh * 2 * (n16 ? 16 : BN));
      float acc[BN];
#pragma unroll
      for (int n = 0; n < BN; ++n) acc[n] = 0.0f;
      for (int kb = 0; kb < kdim / C::BK; ++kb, ++i) {
        const int g = (int)(i % C::NG);
        if (!warp_wait(pfull_bar(g), (i / C::NG) & 1u, args.status, limit)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        // The weight row's scale bytes of four stages per 16-byte read.
        if ((kb & 3) == 0) sc4 = *reinterpret_cast<const uint4*>(srow + kb * 4);
        const uint32_t sw = (kb & 3) == 0 ? sc4.x : (kb & 3) == 1 ? sc4.y : (kb & 3) == 2 ? sc4.z
                                                                                       : sc4.w;
        const uint32_t ta = t_lane + (uint32_t)(g * 4 * BN);
        if (n16) {
          float P[32];
          tmem_ld32(ta, P);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(pempty_bar(g));
          scale_blocks<16>(P, acc, sw, bh, fpanel + (size_t)kb * 4 * BN);
        } else {
          float P[64];
          tmem_ld64(ta, P);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(pempty_bar(g));
          scale_blocks<32>(P, acc, sw, bh, fpanel + (size_t)kb * 4 * BN);
        }
      }
      named_barrier_sync(1, NT);
      if (*abort_flag) break;
      if (lane == 0) mbar_arrive(bempty_bar(p));  // this unit's scale panels are read
      // The two halves' partial sums, added in smem: epi[row][n].
      if (bh == 0) {
#pragma unroll
        for (int n = 0; n < BN; ++n) epi[r * 33 + n] = acc[n];
      }
      named_barrier_sync(1, NT);
      if (bh == 1) {
#pragma unroll
        for (int n = 0; n < BN; ++n) epi[r * 33 + n] += acc[n];
      }
      named_barrier_sync(1, NT);
      if constexpr (GATED) {
        // Thread: token column jj, features 8 fg .. 8 fg + 7 of the unit's 64;
        // a block of 32 features is four neighbouring threads (fg & 3).
        const int jj = et >> 3, fg = et & 7;
        float hv[8];
        float amax = 0.0f;
#pragma unroll
        for (int f = 0; f < 8; ++f) {
          const float gt = epi[(fg * 8 + f) * 33 + jj];
          const float up = epi[(64 + fg * 8 + f) * 33 + jj];
          hv[f] = __fdividef(gt, 1.0f + __expf(-gt)) * up;
          amax = fmaxf(amax, fabsf(hv[f]));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int e = mx_block_exponent(amax);
        const float inv = mx_pow2(-e);
        const uint32_t lo = mx_encode4(hv[0] * inv, hv[1] * inv, hv[2] * inv, hv[3] * inv);
        const uint32_t hi = mx_encode4(hv[4] * inv, hv[5] * inv, hv[6] * inv, hv[7] * inv);
        if (jj < tl.n_valid) {
          uint8_t* out = reinterpret_cast<uint8_t*>(shared ? args.out_shared : args.out);
          uint8_t* osc = shared ? args.out_shared_scales : args.out_scales;
          const int ld = shared ? args.ld_out_shared : args.ld_out_routed;
          const int sko = shared ? args.sko_shared : args.sko_routed;
          const size_t row = (size_t)(shared ? tl.p0 - offs[E] : tl.p0) + jj;
          const int f0 = tl.nb * 64 + fg * 8;
          *reinterpret_cast<uint2*>(out + row * ld + f0) = make_uint2(lo, hi);
          if ((fg & 3) == 0) osc[row * sko + f0 / 32] = (uint8_t)(e + 127);
        }
      } else {
        // Per-token destination rows and gate weights; then thread = output
        // feature r, token columns 16 bh .. 16 bh + 15.
        int32_t* yrow = reinterpret_cast<int32_t*>(epi + 128 * 33);
        float* wt = epi + 128 * 33 + BN;
        for (int j = et; j < tl.n_valid; j += NT) {
          int row;
          float wv;
          if (shared) {
            const int t = tl.p0 - offs[E] + j;
            row = t * args.KP + args.k;
            wv = 1.0f;
          } else {
            const int s = args.gather_idx[tl.p0 + j];
            if ((unsigned)s < (unsigned)(args.T * args.k)) {
              const int t = s / args.k;
              row = t * args.KP + (s - t * args.k);
              wv = args.topk_w[s];
            } else {  // device check: reported; the column goes to row 0 as zeros
              set_status(args.status, MOE_ERR_DEVICE_CHECK);
              row = 0;
              wv = 0.f;
            }
          }
          yrow[j] = row;
          wt[j] = wv;
        }
        named_barrier_sync(1, NT);
        float* Yc = reinterpret_cast<float*>(args.out) + tl.nb * 128 + r;
        const size_t H = (size_t)args.n_out_routed;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          const int j = bh * 16 + n;
          if (j < tl.n_valid) Yc[(size_t)yrow[j] * H] = wt[j] * epi[r * 33 + j];
        }
      }
      named_barrier_sync(1, NT);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// Opt-in shared memory of the current device, looked up once per device.
int smem_optin() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess)
      cache[dev] = v;
  }
  return cache[dev];
}

template <bool GATED, int BN, int STAGES, int CST, int BK>
cudaError_t launch_mx_variant(const MxGemmArgs& a, int num_sms, size_t upper_units,
                              cudaStream_t st) {
  using C = MxCfg<GATED, BN, STAGES, CST, BK>;
  const int sk_max = a.sk_routed > a.sk_shared ? a.sk_routed : a.sk_shared;
  const size_t smem = C::smem_bytes(a.E, sk_max);
  const int optin = smem_optin();
  if (smem > (size_t)optin) return cudaErrorInvalidValue;
  auto fn = mx_gemm_kernel<GATED, BN, STAGES, CST, BK>;
  cudaError_t e = ensure_smem_attr((const void*)fn, (size_t)optin);
  if (e != cudaSuccess) return e;
  size_t grid = (size_t)num_sms;
  if (upper_units < grid) grid = upper_units;
  if (grid == 0) return cudaSuccess;
  return launch_chained(fn, dim3((unsigned)grid), dim3(C::THREADS), smem, st, 1, a);
}

// wide: 256-token tiles with K = 64 stages (token ring of 4 stages of 32 KB,
// code ring of 5 of 8 KB; fewer when the scale panels of a wide K or many
// experts leave no room); otherwise 128-token tiles with K = 128 stages
// (token ring of 4 stages of 32 KB, code ring of 3 of 16 KB; or fewer).
// Decode-sized batches run mx_dec_kernel.
template <bool GATED>
cudaError_t launch_mx(const MxGemmArgs& a, bool wide, int num_sms, size_t ub, cudaStream_t st) {
  const int sk_max = a.sk_routed > a.sk_shared ? a.sk_routed : a.sk_shared;
  const size_t optin = (size_t)smem_optin();
  if (wide) {
    if (MxCfg<GATED, 256, 4, 5, 64>::smem_bytes(a.E, sk_max) <= optin)
      return launch_mx_variant<GATED, 256, 4, 5, 64>(a, num_sms, ub, st);
    if (MxCfg<GATED, 256, 3, 4, 64>::smem_bytes(a.E, sk_max) <= optin)
      return launch_mx_variant<GATED, 256, 3, 4, 64>(a, num_sms, ub, st);
    return launch_mx_variant<GATED, 256, 2, 3, 64>(a, num_sms, ub, st);
  }
  if (MxCfg<GATED, 128, 4, 3, 128>::smem_bytes(a.E, sk_max) <= optin)
    return launch_mx_variant<GATED, 128, 4, 3, 128>(a, num_sms, ub, st);
  if (MxCfg<GATED, 128, 3, 3, 128>::smem_bytes(a.E, sk_max) <= optin)
    return launch_mx_variant<GATED, 128, 3, 3, 128>(a, num_sms, ub, st);
  return launch_mx_variant<GATED, 128, 2, 2, 128>(a, num_sms, ub, st);
}

// 256-token tiles when the experts average at least 256 routed rows (each
// converted weight tile then serves twice the tokens); below that a 256-token
// tile would run half empty and its K = 64 stages cost more per weight byte.
bool mx_wide_tiles(const GemmProblem& p) { return (int64_t)p.T * p.k >= 256 * (int64_t)p.E; }

// The converter kernel's weight-code maps: 64-byte boxes with the 64-byte
// swizzle for K = 64 stages (wide), else 128-byte boxes with the 128-byte one.
bool make_code_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_rows, bool wide) {
  return wide ? make_code_map64(m, base, rows, cols, box_rows)
              : make_tma_map(m, base, MOE_DTYPE_E4M3, rows, cols, box_rows);
}

bool mx_decode_tiles(const GemmProblem& p) {
  return p.tile == MOE_TILE_DECODE || (p.tile == MOE_TILE_AUTO && p.T <= 64);
}

void fill_mx_common(MxGemmArgs& a, const GemmProblem& p, const int32_t* offsets,
                    const int32_t* gather_idx, int* status, int tile_n) {
  a.offsets = offsets;
  a.gather_idx = gather_idx;
  a.status = status;
  a.limit_ns = p.limit_ns;
  a.T = p.T;
  a.k = p.k;
  a.E = p.E;
  a.KP = p.k + (p.Is > 0 ? 1 : 0);
  a.flags = p.flags;
  a.m_lo = 1;
  a.m_hi = 1 << 30;
  a.tile_n = tile_n;
}

}  // namespace

namespace {

template <bool GATED, int STAGES>
cudaError_t launch_mx_dec_variant(const MxGemmArgs& a, int num_sms, size_t upper_units,
                                  cudaStream_t st) {
  using C = MxDecCfg<GATED, STAGES>;
  const int skb_max = a.skb_routed > a.skb_shared ? a.skb_routed : a.skb_shared;
  const int kmax = a.kdim_routed > a.kdim_shared ? a.kdim_routed : a.kdim_shared;
  const size_t smem = C::smem_bytes(a.E, skb_max, kmax / 32);
  const int optin = smem_optin();
  if (smem > (size_t)optin) return cudaErrorInvalidValue;
  auto fn = mx_dec_kernel<GATED, STAGES>;
  cudaError_t e = ensure_smem_attr((const void*)fn, (size_t)optin);
  if (e != cudaSuccess) return e;
  size_t grid = (size_t)num_sms;
  if (upper_units < grid) grid = upper_units;
  if (grid == 0) return cudaSuccess;
  return launch_chained(fn, dim3((unsigned)grid), dim3(C::THREADS), smem, st, 1, a);
}

// The deepest ring of 20 KB stages (8, 6 or 4) that fits next to the scale
// panels of the problem.
template <bool GATED>
cudaError_t launch_mx_dec(const MxGemmArgs& a, int num_sms, size_t ub, cudaStream_t st) {
  const int skb_max = a.skb_routed > a.skb_shared ? a.skb_routed : a.skb_shared;
  const int kmax = a.kdim_routed > a.kdim_shared ? a.kdim_routed : a.kdim_shared;
  const size_t optin = (size_t)smem_optin();
  if (MxDecCfg<GATED, 8>::smem_bytes(a.E, skb_max, kmax / 32) <= optin)
    return launch_mx_dec_variant<GATED, 8>(a, num_sms, ub, st);
  if (MxDecCfg<GATED, 6>::smem_bytes(a.E, skb_max, kmax / 32) <= optin)
    return launch_mx_dec_variant<GATED, 6>(a, num_sms, ub, st);
  return launch_mx_dec_variant<GATED, 4>(a, num_sms, ub, st);
}

}  // namespace

bool mx_uses_decode_kernels(const GemmProblem& p) { return mx_decode_tiles(p); }

cudaError_t launch_mx_dec_swiglu_gemm(const GemmProblem& p, const MxWeights& w,
                                      const MxDecTokens& x, const int32_t* offsets,
                                      const int32_t* gather_idx, const MxDecOut& h, int* status,
                                      cudaStream_t st) {
  const bool has_s = p.Is > 0;
  const int skH = mx_scale_cols(p.H), skI = mx_scale_cols(p.I);
  const int skIs = has_s ? mx_scale_cols(p.Is) : skI;
  MxGemmArgs a;
  memset(&a, 0, sizeof(a));
  const uint64_t R = (uint64_t)p.E * p.I;
  bool ok = make_tma_map(&a.tmA[0], w.gate, MOE_DTYPE_E4M3, R, p.H, 64) &&
            make_tma_map(&a.tmA[1], w.up, MOE_DTYPE_E4M3, R, p.H, 64) &&
            make_scale_map(&a.tmS[0], w.s_gate, R, skH, 64) &&
            make_scale_map(&a.tmS[1], w.s_up, R, skH, 64) &&
            make_b_maps(&a.tmB[0], x.routed, MOE_DTYPE_E4M3, (uint64_t)p.T * p.k, p.H, 32, 16) &&
            make_b_maps(&a.tmB[3], x.shared, MOE_DTYPE_E4M3, p.T, p.H, 32, 16) &&
            make_scale_map(&a.tmSB[0], x.routed_scales, (uint64_t)p.T * p.k, skH, 32) &&
            make_scale_map(&a.tmSB[1], x.shared_scales, p.T, skH, 32);
  if (ok && has_s)
    ok = make_tma_map(&a.tmA[2], w.sh_gate, MOE_DTYPE_E4M3, p.Is, p.H, 64) &&
         make_tma_map(&a.tmA[3], w.sh_up, MOE_DTYPE_E4M3, p.Is, p.H, 64) &&
         make_scale_map(&a.tmS[2], w.sh_s_gate, p.Is, skH, 64) &&
         make_scale_map(&a.tmS[3], w.sh_s_up, p.Is, skH, 64);
  if (!ok) return cudaErrorInvalidValue;
  if (!has_s) {
    a.tmA[2] = a.tmA[0];
    a.tmA[3] = a.tmA[1];
    a.tmS[2] = a.tmS[0];
    a.tmS[3] = a.tmS[1];
  }
  fill_mx_common(a, p, offsets, gather_idx, status, 32);
  a.out = h.routed;
  a.out_shared = h.shared;
  a.out_scales = h.routed_scales;
  a.out_shared_scales = h.shared_scales;
  a.sko_routed = skI;
  a.sko_shared = skIs;
  a.n_out_routed = p.I;
  a.n_out_shared = has_s ? p.Is : 64;
  a.kdim_routed = p.H;
  a.kdim_shared = p.H;
  a.skb_routed = skH;
  a.skb_shared = skH;
  a.ld_out_routed = p.I;
  a.ld_out_shared = has_s ? p.Is : 0;
  const size_t ub = unit_upper_bound(p.T, p.k, p.E, 32, p.I / 64, has_s ? p.Is / 64 : 0);
  return launch_mx_dec<true>(a, p.num_sms, ub, st);
}

cudaError_t launch_mx_dec_down_gemm(const GemmProblem& p, const MxWeights& w,
                                    const MxDecTokens& h, const int32_t* offsets,
                                    const int32_t* gather_idx, const float* topk_w, float* Y,
                                    int* status, cudaStream_t st) {
  const bool has_s = p.Is > 0;
  const int skI = mx_scale_cols(p.I);
  const int skIs = has_s ? mx_scale_cols(p.Is) : skI;
  MxGemmArgs a;
  memset(&a, 0, sizeof(a));
  const uint64_t R = (uint64_t)p.E * p.H;
  bool ok = make_tma_map(&a.tmA[0], w.down, MOE_DTYPE_E4M3, R, p.I, 128) &&
            make_scale_map(&a.tmS[0], w.s_down, R, skI, 128) &&
            make_b_maps(&a.tmB[0], h.routed, MOE_DTYPE_E4M3, (uint64_t)p.T * p.k, p.I, 32, 16) &&
            make_scale_map(&a.tmSB[0], h.routed_scales, (uint64_t)p.T * p.k, skI, 32);
  if (ok && has_s)
    ok = make_tma_map(&a.tmA[2], w.sh_down, MOE_DTYPE_E4M3, p.H, p.Is, 128) &&
         make_scale_map(&a.tmS[2], w.sh_s_down, p.H, skIs, 128) &&
         make_b_maps(&a.tmB[3], h.shared, MOE_DTYPE_E4M3, p.T, p.Is, 32, 16) &&
         make_scale_map(&a.tmSB[1], h.shared_scales, p.T, skIs, 32);
  if (!ok) return cudaErrorInvalidValue;
  if (!has_s) {
    a.tmA[2] = a.tmA[0];
    a.tmS[2] = a.tmS[0];
    for (int i = 0; i < 3; ++i) a.tmB[3 + i] = a.tmB[i];
    a.tmSB[1] = a.tmSB[0];
  }
  a.tmA[1] = a.tmA[0];
  a.tmA[3] = a.tmA[2];
  a.tmS[1] = a.tmS[0];
  a.tmS[3] = a.tmS[2];
  fill_mx_common(a, p, offsets, gather_idx, status, 32);
  a.topk_w = topk_w;
  a.out = Y;
  a.n_out_routed = p.H;
  a.n_out_shared = p.H;
  a.kdim_routed = p.I;
  a.kdim_shared = has_s ? p.Is : p.I;
  a.skb_routed = skI;
  a.skb_shared = skIs;
  const size_t ub = unit_upper_bound(p.T, p.k, p.E, 32, p.H / 128, has_s ? p.H / 128 : 0);
  return launch_mx_dec<false>(a, p.num_sms, ub, st);
}

bool mx_problem_fits(const GemmProblem& p) {
  const size_t optin = (size_t)smem_optin();
  const int skH = mx_scale_cols(p.H), skI = mx_scale_cols(p.I);
  const int skIs = p.Is > 0 ? mx_scale_cols(p.Is) : 0;
  const int skd = skI > skIs ? skI : skIs;
  if (mx_decode_tiles(p)) {
    const int kd = p.I > p.Is ? p.I : p.Is;
    return MxDecCfg<true, 4>::smem_bytes(p.E, skH, p.H / 32) <= optin &&
           MxDecCfg<false, 4>::smem_bytes(p.E, skd, kd / 32) <= optin;
  }
  return MxCfg<true, 256, 2, 3, 64>::smem_bytes(p.E, skH) <= optin &&
         MxCfg<false, 256, 2, 3, 64>::smem_bytes(p.E, skd) <= optin &&
         MxCfg<true, 128, 2, 2, 128>::smem_bytes(p.E, skH) <= optin &&
         MxCfg<false, 128, 2, 2, 128>::smem_bytes(p.E, skd) <= optin;
}

cudaError_t launch_mx_swiglu_gemm(const GemmProblem& p, const MxWeights& w, const void* xq,
                                  const void* xg, const int32_t* offsets,
                                  const int32_t* gather_idx, void* h, void* hs, int* status,
                                  cudaStream_t st) {
  const bool has_s = p.Is > 0;
  if (mx_decode_tiles(p)) return cudaErrorInvalidValue;  // the decode kernels' problems
  const bool wide = mx_wide_tiles(p);
  const int bn = wide ? 256 : 128;
  const uint32_t b1 = bn / 2 < 16 ? 16 : bn / 2;
  const int skH = mx_scale_cols(p.H);
  MxGemmArgs a;
  memset(&a, 0, sizeof(a));
  bool ok = make_code_map(&a.tmA[0], w.gate, (uint64_t)p.E * p.I, p.H, 64, wide) &&
            make_code_map(&a.tmA[1], w.up, (uint64_t)p.E * p.I, p.H, 64, wide) &&
            make_scale_map(&a.tmS[0], w.s_gate, (uint64_t)p.E * p.I, skH, 64) &&
            make_scale_map(&a.tmS[1], w.s_up, (uint64_t)p.E * p.I, skH, 64) &&
            make_b_maps(&a.tmB[0], xg, MOE_DTYPE_BF16, (uint64_t)p.T * p.k, p.H, bn, b1) &&
            make_b_maps(&a.tmB[3], xq, MOE_DTYPE_BF16, p.T, p.H, bn, b1);
  if (ok && has_s)
    ok = make_code_map(&a.tmA[2], w.sh_gate, p.Is, p.H, 64, wide) &&
         make_code_map(&a.tmA[3], w.sh_up, p.Is, p.H, 64, wide) &&
         make_scale_map(&a.tmS[2], w.sh_s_gate, p.Is, skH, 64) &&
         make_scale_map(&a.tmS[3], w.sh_s_up, p.Is, skH, 64);
  if (!ok) return cudaErrorInvalidValue;
  if (!has_s) {
    a.tmA[2] = a.tmA[0];
    a.tmA[3] = a.tmA[1];
    a.tmS[2] = a.tmS[0];
    a.tmS[3] = a.tmS[1];
  }
  fill_mx_common(a, p, offsets, gather_idx, status, bn);
  a.topk_w = nullptr;
  a.out = h;
  a.out_shared = hs;
  a.n_out_routed = p.I;
  a.n_out_shared = has_s ? p.Is : 64;
  a.kdim_routed = p.H;
  a.kdim_shared = p.H;
  a.sk_routed = skH;
  a.sk_shared = skH;
  a.ld_out_routed = p.I;
  a.ld_out_shared = has_s ? p.Is : 0;
  const size_t ub = unit_upper_bound(p.T, p.k, p.E, bn, p.I / 64, has_s ? p.Is / 64 : 0);
  return launch_mx<true>(a, wide, p.num_sms, ub, st);
}

cudaError_t launch_mx_down_gemm(const GemmProblem& p, const MxWeights& w, const void* h,
                                const void* hs, const int32_t* offsets, const int32_t* gather_idx,
                                const float* topk_w, float* Y, int* status, cudaStream_t st) {
  const bool has_s = p.Is > 0;
  if (mx_decode_tiles(p)) return cudaErrorInvalidValue;  // the decode kernels' problems
  const bool wide = mx_wide_tiles(p);
  const int bn = wide ? 256 : 128;
  const uint32_t b1 = bn / 2 < 16 ? 16 : bn / 2;
  const int skI = mx_scale_cols(p.I);
  const int skIs = has_s ? mx_scale_cols(p.Is) : skI;
  MxGemmArgs a;
  memset(&a, 0, sizeof(a));
  bool ok = make_code_map(&a.tmA[0], w.down, (uint64_t)p.E * p.H, p.I, 128, wide) &&
            make_scale_map(&a.tmS[0], w.s_down, (uint64_t)p.E * p.H, skI, 128) &&
            make_b_maps(&a.tmB[0], h, MOE_DTYPE_BF16, (uint64_t)p.T * p.k, p.I, bn, b1);
  if (ok && has_s)
    ok = make_code_map(&a.tmA[2], w.sh_down, p.H, p.Is, 128, wide) &&
         make_scale_map(&a.tmS[2], w.sh_s_down, p.H, skIs, 128) &&
         make_b_maps(&a.tmB[3], hs, MOE_DTYPE_BF16, p.T, p.Is, bn, b1);
  if (!ok) return cudaErrorInvalidValue;
  if (!has_s) {
    a.tmA[2] = a.tmA[0];
    a.tmS[2] = a.tmS[0];
    for (int i = 0; i < 3; ++i) a.tmB[3 + i] = a.tmB[i];
  }
  a.tmA[1] = a.tmA[0];
  a.tmA[3] = a.tmA[2];
  a.tmS[1] = a.tmS[0];
  a.tmS[3] = a.tmS[2];
  fill_mx_common(a, p, offsets, gather_idx, status, bn);
  a.topk_w = topk_w;
  a.out = Y;
  a.out_shared = nullptr;
  a.n_out_routed = p.H;
  a.n_out_shared = p.H;
  a.kdim_routed = p.I;
  a.kdim_shared = has_s ? p.Is : p.I;
  a.sk_routed = skI;
  a.sk_shared = skIs;
  a.ld_out_routed = p.H;
  a.ld_out_shared = p.H;
  const size_t ub = unit_upper_bound(p.T, p.k, p.E, bn, p.H / 128, has_s ? p.H / 128 : 0);
  return launch_mx<false>(a, wide, p.num_sms, ub, st);
}

}  // namespace moe
