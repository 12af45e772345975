// Internal launch functions of the kernels behind the C ABI (not exported).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe_api.h"

namespace moe {

// TMA tensor map of a row-major [rows][cols] matrix of MOE_DTYPE_* elements:
// boxes of 128 bytes of columns x box_rows rows, 128-byte swizzle, zero fill
// out of bounds (grouped_gemm.cu). False if the driver entry point is missing
// or the encoder rejects the shape.
bool make_tma_map(CUtensorMap* m, const void* base, int dtype, uint64_t rows, uint64_t cols,
                  uint32_t box_rows);
// Tensor map of E4M3 codes [rows][cols]: boxes of 64 bytes x box_rows rows,
// 64-byte swizzle.
bool make_code_map64(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows);
// Tensor map of a uint8 [rows][cols] matrix (cols a multiple of 16) whose box
// is box_cols bytes (0: whole rows; a multiple of 16, at most 256) of box_rows
// rows, no swizzle.
bool make_scale_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t cols,
                    uint32_t box_rows, uint32_t box_cols = 0);
// Tensor maps of a tiled token operand [rows][cols]: boxes of b_rows, box1 and
// 16 rows.
bool make_b_maps(CUtensorMap* m, const void* base, int dtype, uint64_t rows, uint64_t cols,
                 uint32_t b_rows, uint32_t box1);
// Upper bound of the unit count of one grouped-GEMM launch (token tiles of
// tile_n rows, routed_blocks / shared_blocks feature blocks per group).
size_t unit_upper_bound(int T, int k, int E, int tile_n, int routed_blocks, int shared_blocks);
// Raise a kernel's dynamic shared-memory limit to smem once per device.
cudaError_t ensure_smem_attr(const void* fn, size_t smem);

// Router (router.cu).
// Slices S of H whose partial logits the router writes (S == 1: final logits).
int router_split_count(int dtype, int64_t T, int64_t H, int64_t E, int num_sms);
// bf16: tensor cores (status/limit_ns bound its waits); fp32: CUDA cores.
cudaError_t launch_router_logits(int dtype, const void* x, const void* Wr, const float* bias,
                                 int T, int H, int E, int S, float* out_partials, int* status,
                                 unsigned long long limit_ns, cudaStream_t st);
cudaError_t launch_logits_reduce(const float* partials, int S, int T, int E, const float* bias,
                                 float* logits, int num_sms, cudaStream_t st);
// n_group <= 1: plain top-k; else the top-k limited to the best topk_group of
// n_group contiguous expert groups.
cudaError_t launch_route(const float* src, int S, const float* bias, int T, int E, int k,
                         int renorm, int n_group, int topk_group, float* logits_out,
                         int32_t* ids, float* w, cudaStream_t st);

// Permutation (permute.cu).
size_t permute_smem_bytes(int E);
// Workspace bytes of per-chunk counts the grid-wide variant needs (0 when one
// CTA does the whole permutation).
size_t permute_scratch_bytes(int64_t T, int64_t E, int64_t k);
cudaError_t launch_permute(const int32_t* ids, int T, int E, int k, int has_shared,
                           int32_t* offsets, int32_t* gather_idx, int32_t* slot_pos, int* status,
                           int32_t* chunk_hist, cudaStream_t st);

// Dispatch copy of the routed token rows into expert order (permute.cu).
// Row slot_pos[s] of xg = x[s / k] for the P = T*k slots (slot order); a
// position beyond P sets MOE_ERR_DEVICE_CHECK in *status and is skipped.
cudaError_t launch_gather_rows(const void* x, const int32_t* slot_pos, int P, int k,
                               size_t row_bytes, void* xg, int* status, int num_sms,
                               cudaStream_t st);

// Grouped GEMMs (grouped_gemm.cu).
struct GemmProblem {
  int dtype;  // MOE_DTYPE_*
  int tile;   // moe_tile: AUTO chooses per expert from its row count
  int T, H, E, k, I, Is;
  unsigned flags;
  unsigned long long limit_ns;
  int num_sms;
};
// xg: the routed token rows in expert order ([T*k][H], from launch_gather_rows);
// required when gemm_needs_expert_order_copy(p) (128/256-token tiles may run),
// ignored otherwise (32-token tiles gather rows in the GEMM's own loads).
bool gemm_needs_expert_order_copy(const GemmProblem& p);
// True when both GEMMs run the 32-token decode kernels (gather4 token rows).
bool gemm_uses_decode_tiles(const GemmProblem& p);
// Per-row power-of-two scales of E4M3 operands (dtype MOE_DTYPE_E4M3 only):
// a[0..3] = gate, up, shared gate, shared up rows (gated GEMM) or a[0] = W_down,
// a[2] = shared W_down rows (down GEMM); b[0] = x rows by token (gated) or h
// rows by position (down), b[1] = h_shared rows by token (down).
struct GemmScales {
  const float* a[4];
  const float* b[2];
};
cudaError_t launch_swiglu_gemm(const GemmProblem& p, const void* x, const void* xg,
                               const int32_t* offsets, const int32_t* gather_idx, const void* Wg,
                               const void* Wu, const void* Wsg, const void* Wsu, void* h, void* hs,
                               int* status, cudaStream_t st, const GemmScales* sc = nullptr);
cudaError_t launch_down_gemm(const GemmProblem& p, const void* h, const void* hs,
                             const int32_t* offsets, const int32_t* gather_idx,
                             const float* topk_w, const void* Wd, const void* Wsd, float* Y,
                             int* status, cudaStream_t st, const GemmScales* sc = nullptr);
bool tensor_map_encoder_available();

// Entry-point helpers (moe_api.cu), shared by every C ABI call so that all of
// them validate and describe a problem the same way.
// SM count of the current device, cached per device under a mutex.
int sm_count();
// Argument checks of a moe_problem (shapes, dtype, tile, the int32 index
// ranges the kernels rely on); MOE_OK or the error to return before any launch.
moe_status check_problem(const moe_problem* pb, bool allow_quantized = false);
// The grouped-GEMM description of a checked problem.
GemmProblem gemm_problem(const moe_problem& p);

// Single-launch decode path (fused_decode.cu): the whole layer in one
// cooperative persistent kernel for decode-sized batches. Pointers as in
// moe_forward; grid_ctr (zero at launch) and unit_done ([E+1]) are workspace.
struct FusedDecodeIO {
  const void* x;
  const void* Wr;
  const float* bias;
  int renorm, n_group, topk_group, out_f32;
  const void *Wg, *Wu, *Wd, *Wsg, *Wsu, *Wsd;
  float* logits;
  int32_t* ids;
  float* w;
  int32_t *offsets, *gather_idx, *slot_pos;
  void *h, *hs;
  float* Y;
  void* y;
  int* status;
  int* grid_ctr;
  int* unit_done;
  float* router_part;  // [8][T][E]: the router's partial sums over slices of H
};
// True when the problem runs the decode tiles, fits one CTA per SM with a CTA
// per token, and the device supports cooperative launches.
bool fused_decode_supported(const GemmProblem& p);
cudaError_t launch_fused_decode(const GemmProblem& p, const FusedDecodeIO& io, cudaStream_t st);

// Row quantization to E4M3 with a power-of-two scale per row (quantize.cu):
// src [rows][cols] of MOE_DTYPE_BF16 or MOE_DTYPE_F32, cols a multiple of 16.
cudaError_t launch_quantize_rows(int dtype, const void* src, int64_t rows, int64_t cols,
                                 uint8_t* q, float* scale, int num_sms, cudaStream_t st);

// MXFP8 (quantize_mx.cu): blocks of 32 elements along each row, one E8M0
// scale byte per block (rows of mx_scale_cols(cols) bytes, zero padded).
// launch_quantize_mx: src [rows][cols] bf16 or fp32 -> codes + scales;
// launch_qdq_mx: bf16 src -> the bf16 value of every element after
// quantization (the MXFP8 layer's token rows). cols a multiple of 32.
cudaError_t launch_quantize_mx(int dtype, const void* src, int64_t rows, int64_t cols,
                               uint8_t* q, uint8_t* scales, int num_sms, cudaStream_t st);
cudaError_t launch_qdq_mx(const void* src, int64_t rows, int64_t cols, void* out, int num_sms,
                          cudaStream_t st);
// The decode-sized MXFP8 layer's token operand: bf16 x [T][H] -> codes and scale
// rows of every routed slot at its position (xgq [T*k][H], xgs [T*k][sk]), and
// in token order (xq, xs; skipped when null). A position beyond T*k sets
// MOE_ERR_DEVICE_CHECK in *status and is skipped.
cudaError_t launch_quantize_dispatch_mx(const void* x, const int32_t* slot_pos, int T, int k,
                                       int H, uint8_t* xgq, uint8_t* xgs, uint8_t* xq, uint8_t* xs,
                                       int* status, int num_sms, cudaStream_t st);

// MXFP8 grouped GEMMs (grouped_gemm_mx.cu). Weight codes [rows][K] with
// their scale rows; the shared expert's (sh_*) are null without one.
struct MxWeights {
  const uint8_t *gate, *s_gate, *up, *s_up, *down, *s_down;
  const uint8_t *sh_gate, *sh_s_gate, *sh_up, *sh_s_up, *sh_down, *sh_s_down;
};
// True when both MXFP8 GEMMs of the problem fit the device's shared memory.
bool mx_problem_fits(const GemmProblem& p);
// Batches beyond the decode size (128-token tiles; decode-sized problems are
// refused here and run launch_mx_dec_*): xq: the quantized token rows [T][H]
// (bf16 values); xg: their expert-ordered copy [T*k][H]; h, hs bf16 outputs
// holding MXFP8 values.
cudaError_t launch_mx_swiglu_gemm(const GemmProblem& p, const MxWeights& w, const void* xq,
                                  const void* xg, const int32_t* offsets,
                                  const int32_t* gather_idx, void* h, void* hs, int* status,
                                  cudaStream_t st);
cudaError_t launch_mx_down_gemm(const GemmProblem& p, const MxWeights& w, const void* h,
                                const void* hs, const int32_t* offsets, const int32_t* gather_idx,
                                const float* topk_w, float* Y, int* status, cudaStream_t st);
// Decode-sized problems (32-token tiles) run the E4M3-MMA kernels instead:
// token operands are MXFP8 codes with scale rows; the gate/up GEMM writes h
// and h_shared the same way.
bool mx_uses_decode_kernels(const GemmProblem& p);
struct MxDecTokens {
  const uint8_t *routed, *routed_scales;  // rows by position [T*k]
  const uint8_t *shared, *shared_scales;  // rows by token [T] (x, or h_shared)
};
struct MxDecOut {
  uint8_t *routed, *routed_scales, *shared, *shared_scales;
};
cudaError_t launch_mx_dec_swiglu_gemm(const GemmProblem& p, const MxWeights& w,
                                      const MxDecTokens& x, const int32_t* offsets,
                                      const int32_t* gather_idx, const MxDecOut& h, int* status,
                                      cudaStream_t st);
cudaError_t launch_mx_dec_down_gemm(const GemmProblem& p, const MxWeights& w,
                                    const MxDecTokens& h, const int32_t* offsets,
                                    const int32_t* gather_idx, const float* topk_w, float* Y,
                                    int* status, cudaStream_t st);

// Combine (combine.cu): y[t] = sum_j Y[t][j] for j < KP, rank order.
cudaError_t launch_combine(int dtype, const float* Y, int T, int H, int KP, void* y,
                           int num_sms, cudaStream_t st);

}  // namespace moe
