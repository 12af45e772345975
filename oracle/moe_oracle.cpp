// CPU oracle for the Mixture-of-Experts FFN layer forward pass.
//
// TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
// CPU-baseline leg may load this library. It shares no code with the CUDA path
// and neither side includes the other.
//
// It is the plain definition, written as slow loops in the order the pages
// state the layer:
//   1. router logits            l[t][e] = sum_h x[t][h] * Wr[e][h] (+ b[e])
//      ("Lower latency and higher throughput with multi-node DeepSeek
//      deployment", five-stage layer breakdown: the "Gate" ends stage 2).
//   2. top-k on the logits, lowest expert index first among equals, then the
//      softmax gate weights, renormalised over the k chosen experts
//      (same page, section "MoE Router": top-K indices and scores); optionally
//      limited to the best topk_group of n_group expert groups (the same
//      section's DeepSeek form of the router).
//   3. a stable counting sort of the (token, rank) slots by expert: per-expert
//      counts, offsets and a unique position for every slot ("CuTeDSL at
//      Perplexity", section "Mixture-of-Experts Dispatch/Combine", "Local").
//   4. per routed position, the SwiGLU expert FFN: silu(x Wg^T) * (x Wu^T),
//      then the down projection (Qwen3.5-397B on TPU v7x write-up, section
//      4.2.2: gate and up projections with the SwiGLU activation fused).
//   5. the gate-weighted sum of each token's expert outputs, plus the shared
//      expert's output with weight 1 (DeepSeek page, "Expert Parallelism").
//
// Precision: all data are fp32 (bf16 inputs are widened exactly by the
// caller); every sum is accumulated in fp64 in natural index order and rounded
// to fp32 where a stage stores its result (logits, weights, h, y). Selection
// (top-k) compares the stored fp32 logits.
//
// Parity pins (tests/test_oracle.py, CPU only): float64 library matmul for
// the logits; a stable library sort for top-k ids; softmax identities for the
// weights; bijection / stability / library argsort for the permutation;
// brute-force dense evaluation of every expert, the k=E uniform-weight mean of
// experts, the E=1 dense FFN in torch float64, token-permutation equivariance,
// and a hand-derived closed-form case (tests/golden/).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

inline double silu(double z) { return z / (1.0 + std::exp(-z)); }

// One routed or shared FFN evaluation for one token row.
// Wg, Wu: [I][H]; Wd: [H][I]. h_out (nullable) receives fp32 h; o_out: [H] fp64.
void expert_ffn(const float* xr, const float* Wg, const float* Wu, const float* Wd,
                int64_t H, int64_t I, float* h_out, double* o_out) {
  std::vector<float> h(I);
  for (int64_t i = 0; i < I; ++i) {
    const float* wg = Wg + i * H;
    const float* wu = Wu + i * H;
    double g = 0.0, u = 0.0;
    for (int64_t c = 0; c < H; ++c) {
      g += (double)xr[c] * (double)wg[c];
      u += (double)xr[c] * (double)wu[c];
    }
    h[i] = (float)(silu(g) * u);
  }
  if (h_out) std::memcpy(h_out, h.data(), sizeof(float) * I);
  if (o_out) {
    for (int64_t c = 0; c < H; ++c) {
      const float* wd = Wd + c * I;
      double o = 0.0;
      for (int64_t i = 0; i < I; ++i) o += (double)h[i] * (double)wd[i];
      o_out[c] = o;
    }
  }
}

// ---------------------------------------------------------------- FP8 rows
// The FP8 expert path stores a matrix as E4M3 codes with one power-of-two
// scale per row (the microscaling idea of "Hosting Qwen on Blackwell": scale
// factors are exact powers of two, so scaling never rounds).
//
// E4M3 (OCP 8-bit floating point): sign bit, 4 exponent bits with bias 7, 3
// mantissa bits. Exponent field 0 holds the subnormals m/8 * 2^-6. There are no
// infinities; S.1111.111 is NaN, so the largest finite magnitude is
// 1.75 * 2^8 = 448.
double e4m3_decode_one(uint8_t c) {
  const int s = c >> 7, ef = (c >> 3) & 15, m = c & 7;
  if (ef == 15 && m == 7) return std::nan("");
  const double mag = ef == 0 ? std::ldexp((double)m / 8.0, -6)
                             : std::ldexp(1.0 + (double)m / 8.0, ef - 7);
  return s ? -mag : mag;
}

// Nearest E4M3 value to v, ties to the even mantissa; |v| beyond 448 gives
// 448 (callers scale rows so that this never happens).
uint8_t e4m3_encode_one(float v) {
  const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  double a = std::fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;
  // Spacing of the representable magnitudes around a: 2^(E-3) for a in
  // [2^E, 2^(E+1)), E >= -6; 2^-9 below 2^-6 (subnormals).
  int E = -6;
  if (a >= std::ldexp(1.0, -6)) {
    int e2;
    std::frexp(a, &e2);  // a = f * 2^e2, f in [0.5, 1)
    E = e2 - 1;
  }
  const double ulp = std::ldexp(1.0, E - 3);
  double n = std::floor(a / ulp);  // exact: a / ulp is a power-of-two scaling
  const double rem = a / ulp - n;
  if (rem > 0.5 || (rem == 0.5 && std::fmod(n, 2.0) != 0.0)) n += 1.0;
  const double r = n * ulp;  // the rounded magnitude
  if (r >= 448.0) return sign | 0x7E;
  if (r < std::ldexp(1.0, -6)) return sign | (uint8_t)n;  // subnormal: m = n
  int e2;
  const double f = std::frexp(r, &e2);  // r = f * 2^e2
  const int ef = e2 - 1 + 7;
  const int m = (int)std::lround((2.0 * f - 1.0) * 8.0);
  return sign | (uint8_t)((ef << 3) | m);
}

}  // namespace

extern "C" {

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

// Step 1: logits [T][E] = x [T][H] . Wr[E][H]^T (+ bias[E]); fp64 sums, fp32 out.
void oracle_router_logits(const float* x, const float* Wr, const float* bias,
                          int64_t T, int64_t H, int64_t E, float* logits) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t e = 0; e < E; ++e) {
      double s = 0.0;
      for (int64_t c = 0; c < H; ++c) s += (double)x[t * H + c] * (double)Wr[e * H + c];
      if (bias) s += (double)bias[e];
      logits[t * E + e] = (float)s;
    }
  }
}

// Step 2: for each token, k rounds of "largest not yet chosen logit, lowest
// index among equals"; ids come out in descending score order. Weights are
// p_e = exp(l_e - l_max); S = sum over the chosen p (renorm != 0) or over all E
// (renorm == 0); w = p / S.
void oracle_route(const float* logits, int64_t T, int64_t E, int64_t k, int renorm,
                  int32_t* ids, float* w) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    std::vector<char> taken(E, 0);
    for (int64_t r = 0; r < k; ++r) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e;  // strict '>' keeps the lower index
      }
      taken[best] = 1;
      ids[t * k + r] = (int32_t)best;
    }
    const double m = (double)l[ids[t * k]];
    double S = 0.0;
    if (renorm) {
      for (int64_t r = 0; r < k; ++r) S += std::exp((double)l[ids[t * k + r]] - m);
    } else {
      for (int64_t e = 0; e < E; ++e) S += std::exp((double)l[e] - m);
    }
    for (int64_t r = 0; r < k; ++r)
      w[t * k + r] = (float)(std::exp((double)l[ids[t * k + r]] - m) / S);
  }
}

// Step 2, group-limited form ("MoE Router" section of the DeepSeek page: the
// Mixtral router is the DeepSeek router whose top-K group is the group of all
// experts). The E experts form n_group contiguous groups of E / n_group. For
// each token: a group's score is the largest logit in it; the topk_group
// groups with the largest scores are kept (lower group index among equals);
// then k rounds of "largest not yet chosen logit among the kept groups, lowest
// index among equals". Weights as in oracle_route, from the unmasked logits
// (renorm == 0: the softmax over all E). n_group <= 1 is oracle_route.
void oracle_route_grouped(const float* logits, int64_t T, int64_t E, int64_t k, int renorm,
                          int64_t n_group, int64_t topk_group, int32_t* ids, float* w) {
  if (n_group <= 1) {
    oracle_route(logits, T, E, k, renorm, ids, w);
    return;
  }
  const int64_t G = E / n_group;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    std::vector<float> score(n_group);
    for (int64_t j = 0; j < n_group; ++j) {
      float best = l[j * G];
      for (int64_t e = j * G + 1; e < (j + 1) * G; ++e)
        if (l[e] > best) best = l[e];
      score[j] = best;
    }
    std::vector<char> kept(n_group, 0);
    for (int64_t r = 0; r < topk_group; ++r) {
      int64_t bj = -1;
      for (int64_t j = 0; j < n_group; ++j) {
        if (kept[j]) continue;
        if (bj < 0 || score[j] > score[bj]) bj = j;  // strict '>' keeps the lower index
      }
      kept[bj] = 1;
    }
    std::vector<char> taken(E, 0);
    for (int64_t r = 0; r < k; ++r) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e) {
        if (taken[e] || !kept[e / G]) continue;
        if (best < 0 || l[e] > l[best]) best = e;
      }
      taken[best] = 1;
      ids[t * k + r] = (int32_t)best;
    }
    const double m = (double)l[ids[t * k]];
    double S = 0.0;
    if (renorm) {
      for (int64_t r = 0; r < k; ++r) S += std::exp((double)l[ids[t * k + r]] - m);
    } else {
      for (int64_t e = 0; e < E; ++e) S += std::exp((double)l[e] - m);
    }
    for (int64_t r = 0; r < k; ++r)
      w[t * k + r] = (float)(std::exp((double)l[ids[t * k + r]] - m) / S);
  }
}

// Step 3: counting sort of slots s = t*k + r by expert, stable in s.
// offsets[0..E] = exclusive prefix of the counts; offsets[E+1] = offsets[E]
// + (has_shared ? T : 0) closes the shared segment, whose position T*k + t is
// token t. gather_idx[p] = slot at position p; slot_pos[s] = position of slot s.
void oracle_permute(const int32_t* ids, int64_t T, int64_t E, int64_t k, int has_shared,
                    int32_t* offsets, int32_t* gather_idx, int32_t* slot_pos) {
  std::vector<int64_t> cnt(E, 0);
  for (int64_t s = 0; s < T * k; ++s) cnt[ids[s]] += 1;
  offsets[0] = 0;
  for (int64_t e = 0; e < E; ++e) offsets[e + 1] = (int32_t)(offsets[e] + cnt[e]);
  offsets[E + 1] = (int32_t)(offsets[E] + (has_shared ? T : 0));
  std::vector<int64_t> fill(E, 0);
  for (int64_t s = 0; s < T * k; ++s) {
    const int64_t e = ids[s];
    const int64_t p = offsets[e] + fill[e]++;
    gather_idx[p] = (int32_t)s;
    slot_pos[s] = (int32_t)p;
  }
}

// Step 4a: h for every routed position (and the shared rows). x [T][H];
// Wg, Wu [E][I][H]; h [T*k][I]; shared: Wsg, Wsu [Is][H], hs [T][Is].
void oracle_expert_h(const float* x, const int32_t* offsets, const int32_t* gather_idx,
                     const float* Wg, const float* Wu, int64_t T, int64_t H, int64_t E,
                     int64_t k, int64_t I, float* h, const float* Wsg, const float* Wsu,
                     int64_t Is, float* hs) {
  const int64_t P = (int64_t)offsets[E];
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t p = 0; p < P; ++p) {
    int64_t e = 0;
    while (!(p >= offsets[e] && p < offsets[e + 1])) ++e;
    const int64_t t = gather_idx[p] / k;
    expert_ffn(x + t * H, Wg + e * I * H, Wu + e * I * H, nullptr, H, I, h + p * I, nullptr);
  }
  if (Is > 0 && hs) {
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t)
      expert_ffn(x + t * H, Wsg, Wsu, nullptr, H, Is, hs + t * Is, nullptr);
  }
}

// Step 4b + 5 from given h: y[t][c] = sum_r w[t][r] * (h[p] . Wd[e][c][:]) with
// p = slot_pos[t*k + r], plus (hs[t] . Wsd[c][:]) when Is > 0. fp64 sums.
void oracle_down_combine(const float* h, const int32_t* offsets, const int32_t* slot_pos,
                         const int32_t* ids, const float* w, const float* Wd, int64_t T,
                         int64_t H, int64_t E, int64_t k, int64_t I, const float* hs,
                         const float* Wsd, int64_t Is, float* y) {
  (void)offsets;
  (void)E;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < T; ++t) {
    std::vector<double> acc(H, 0.0);
    for (int64_t r = 0; r < k; ++r) {
      const int64_t s = t * k + r;
      const int64_t p = slot_pos[s];
      const int64_t e = ids[s];
      const float* hp = h + p * I;
      const float* wd = Wd + e * H * I;
      for (int64_t c = 0; c < H; ++c) {
        double o = 0.0;
        for (int64_t i = 0; i < I; ++i) o += (double)hp[i] * (double)wd[c * I + i];
        acc[c] += (double)w[s] * o;
      }
    }
    if (Is > 0 && hs) {
      const float* hp = hs + t * Is;
      for (int64_t c = 0; c < H; ++c) {
        double o = 0.0;
        for (int64_t i = 0; i < Is; ++i) o += (double)hp[i] * (double)Wsd[c * Is + i];
        acc[c] += o;
      }
    }
    for (int64_t c = 0; c < H; ++c) y[t * H + c] = (float)acc[c];
  }
}

// Steps 4 + 5 with the routing given: y [T][H] from x, ids, w and the weights.
// Each token is evaluated on its own; nothing is shared between tokens.
void oracle_ffn_combine(const float* x, const int32_t* ids, const float* w, const float* Wg,
                        const float* Wu, const float* Wd, int64_t T, int64_t H, int64_t E,
                        int64_t k, int64_t I, const float* Wsg, const float* Wsu,
                        const float* Wsd, int64_t Is, float* y) {
  (void)E;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < T; ++t) {
    std::vector<double> acc(H, 0.0), o(H);
    for (int64_t r = 0; r < k; ++r) {
      const int64_t e = ids[t * k + r];
      expert_ffn(x + t * H, Wg + e * I * H, Wu + e * I * H, Wd + e * H * I, H, I, nullptr,
                 o.data());
      for (int64_t c = 0; c < H; ++c) acc[c] += (double)w[t * k + r] * o[c];
    }
    if (Is > 0) {
      expert_ffn(x + t * H, Wsg, Wsu, Wsd, H, Is, nullptr, o.data());
      for (int64_t c = 0; c < H; ++c) acc[c] += o[c];
    }
    for (int64_t c = 0; c < H; ++c) y[t * H + c] = (float)acc[c];
  }
}

void oracle_e4m3_decode(const uint8_t* codes, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (float)e4m3_decode_one(codes[i]);
}

void oracle_e4m3_encode(const float* v, int64_t n, uint8_t* codes) {
  for (int64_t i = 0; i < n; ++i) codes[i] = e4m3_encode_one(v[i]);
}

// Row quantization: scale = 2^e with e the smallest integer such that
// max_i |src[r][i]| <= 448 * 2^e (e >= -126; e = 0 for a row of zeros), then
// q[r][i] = E4M3(src[r][i] / 2^e), rounded to nearest even. Dividing by a
// power of two is exact, so dequantization is q * scale.
void oracle_quantize_rows_e4m3(const float* src, int64_t rows, int64_t cols, uint8_t* q,
                               float* scale) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const float* v = src + r * cols;
    double amax = 0.0;
    for (int64_t i = 0; i < cols; ++i) amax = std::fmax(amax, std::fabs((double)v[i]));
    int e = 0;
    if (amax > 0.0) {
      int e2;
      const double f = std::frexp(amax, &e2);  // amax = (2f) * 2^(e2 - 1), 2f in [1, 2)
      const int E = e2 - 1;
      e = (2.0 * f <= 1.75) ? E - 8 : E - 7;
      if (e < -126) e = -126;
    }
    scale[r] = std::ldexp(1.0f, e);
    for (int64_t i = 0; i < cols; ++i)
      q[r * cols + i] = e4m3_encode_one(std::ldexp(v[i], -e));
  }
}

// MXFP8 block quantization ("Hosting Qwen on Blackwell", quantization
// section: Qwen3-235B served with MXFP8 microscaled weights; "CuTeDSL at
// Perplexity", Blackwell quantization paragraph: the absolute maximum over 32
// elements). Each row is cut into blocks of 32 consecutive elements; a block's
// scale is the power of two X = 2^e with e = floor(log2(amax)) - 8 (8 is the
// exponent of E4M3's largest power of two, 256; the Microscaling format's
// rule), held in [-127, 127], and e = -127 for a block of zeros. The scale is
// stored as the unsigned exponent byte e + 127 (E8M0); the elements are the
// E4M3 codes of v / X, nearest even, saturating at 448 (v / X lies in
// [256, 512) for the block's largest element, so values above 448 are
// clamped). Dividing by a power of two is exact, so a value decodes as
// code * X. scales has sk bytes per row (sk >= cols / 32); bytes past the
// row's cols / 32 blocks are zero.
void oracle_quantize_mx(const float* src, int64_t rows, int64_t cols, int64_t sk, uint8_t* q,
                        uint8_t* scales) {
  const int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t j = 0; j < sk; ++j) scales[r * sk + j] = 0;
    for (int64_t b = 0; b < nb; ++b) {
      const float* v = src + r * cols + b * 32;
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) amax = std::fmax(amax, std::fabs((double)v[i]));
      int e = -127;
      if (amax > 0.0) {
        int e2;
        std::frexp(amax, &e2);  // amax = f * 2^e2, f in [0.5, 1): floor(log2) = e2 - 1
        e = e2 - 1 - 8;
        if (e < -127) e = -127;
        if (e > 127) e = 127;
      }
      scales[r * sk + b] = (uint8_t)(e + 127);
      for (int i = 0; i < 32; ++i)
        q[r * cols + b * 32 + i] = e4m3_encode_one(std::ldexp(v[i], -e));
    }
  }
}

// bfloat16 rounding (nearest, ties to even) of fp32 values, returned as fp32.
void oracle_bf16_round(const float* src, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) {
    uint32_t u;
    std::memcpy(&u, &src[i], 4);
    const uint32_t lsb = (u >> 16) & 1u;
    u = (u + 0x7FFFu + lsb) & 0xFFFF0000u;
    std::memcpy(&out[i], &u, 4);
  }
}


// The whole layer: steps 1-5. Every intermediate output pointer is nullable.
void oracle_moe_forward(const float* x, const float* Wr, const float* bias, const float* Wg,
                        const float* Wu, const float* Wd, const float* Wsg, const float* Wsu,
                        const float* Wsd, int64_t T, int64_t H, int64_t E, int64_t k,
                        int64_t I, int64_t Is, int renorm, float* y, float* logits_out,
                        int32_t* ids_out, float* w_out) {
  std::vector<float> logits(T * E), w(T * k);
  std::vector<int32_t> ids(T * k);
  oracle_router_logits(x, Wr, bias, T, H, E, logits.data());
  oracle_route(logits.data(), T, E, k, renorm, ids.data(), w.data());
  oracle_ffn_combine(x, ids.data(), w.data(), Wg, Wu, Wd, T, H, E, k, I, Wsg, Wsu, Wsd, Is, y);
  if (logits_out) std::memcpy(logits_out, logits.data(), sizeof(float) * T * E);
  if (ids_out) std::memcpy(ids_out, ids.data(), sizeof(int32_t) * T * k);
  if (w_out) std::memcpy(w_out, w.data(), sizeof(float) * T * k);
}

}  // extern "C"
