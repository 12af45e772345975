/*
 * moe_api.h — C ABI of the GB300 Mixture-of-Experts FFN layer forward pass.
 *
 * The layer (per token t, with x[t] its hidden row):
 *   logits[t][e] = x[t] . W_router[e] (+ router_bias[e])
 *   ids[t][0..k)  = the k largest logits, descending, lowest index among equals
 *   w[t][r]       = exp(l_{ids[t][r]} - l_max) / S, S summed over the k chosen
 *                   experts (renorm = 1) or over all E experts (renorm = 0)
 *   y[t]          = sum_r w[t][r] * FFN_{ids[t][r]}(x[t])  (+ FFN_shared(x[t]))
 *   FFN_e(v)      = W_down[e] (silu(W_gate[e] v) * (W_up[e] v)),
 *                   silu(z) = z / (1 + exp(-z))
 * Sources: "Lower latency and higher throughput with multi-node DeepSeek
 * deployment" (Perplexity blog; sections "Expert Parallelism", "MoE Router",
 * "GroupGEMM"), "CuTeDSL at Perplexity" (section "Mixture-of-Experts
 * Dispatch/Combine", "Local"), and the Qwen3.5-397B on TPU v7x write-up
 * (section 4.2.1 ragged gather, section 4.2.2 grouped GEMM with fused SwiGLU).
 *
 * Conventions for every call:
 *  - Pointers are DEVICE pointers owned by the caller, unless stated. The library
 *    allocates no device memory; scratch comes from `workspace`, whose size is
 *    given by moe_workspace_size(). Every pointer must be 16-byte aligned.
 *  - Layouts are contiguous row-major: x [T][H]; W_router [E][H];
 *    W_gate, W_up [E][I][H]; W_down [E][H][I]; shared expert Ws_gate, Ws_up
 *    [I_shared][H], Ws_down [H][I_shared]; y [T][H]. Both expert GEMMs are thus
 *    K-major (nn.Linear "out x in" per expert).
 *  - x, the weights, h and y share the problem's dtype (bf16, or fp32 which the
 *    tensor cores consume as tf32). logits and gate weights are fp32; ids,
 *    offsets and indices are int32.
 *  - Shapes: 1 <= k <= E <= 1024, k <= 32; H a multiple of 128; I and I_shared
 *    multiples of 64; T*k and T*(k+1) below 2^31.
 *  - Argument errors are detected on the host before any launch and returned
 *    as MOE_ERR_*; outputs are then untouched. T == 0 is MOE_OK.
 *  - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream); no call synchronises except
 *    moe_get_device_status().
 *  - Asynchronous device conditions (a bounded wait that ran out, a failed
 *    device-side check: an expert id, offset, gather index or slot position
 *    out of range; the access is then skipped or kept inside the buffers) are
 *    recorded in a status word at the start of the
 *    workspace and read with moe_get_device_status(). The word is sticky: once
 *    set, later kernels that see it give up early. moe_forward() clears it
 *    when it starts; the sub-calls do not (use moe_reset_device_status()).
 *    Kernels never trap.
 *  - Results are bitwise reproducible run to run: no floating-point atomics,
 *    fixed reduction orders.
 *  - Thread-compatible: calls on distinct workspaces may run concurrently.
 *    Global state: a per-device cache (SM count, kernel attributes, the
 *    address of the scratch array below) guarded by a mutex, and the one
 *    static scratch array of moe_down_combine_noalloc per device, which every
 *    call of that function uses: its calls must not overlap on one device
 *    (the caller serialises them); the other calls never touch it.
 */
#ifndef MOE_API_H_
#define MOE_API_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* bad pointer, shape, alignment or dtype */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but not supported by the library or device */
  MOE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 5,      /* (device status) a bounded wait ran out */
  MOE_ERR_DEVICE_CHECK = 6  /* (device status) a device-side check failed */
} moe_status;

/* MOE_DTYPE_E4M3: bf16 activations with E4M3 expert weights, one power-of-two
 * scale per weight row (moe_quantize_rows_e4m3); only moe_forward_fp8 takes it.
 * MOE_DTYPE_MXFP8: bf16 activations with MXFP8 expert weights, E4M3 codes with
 * one E8M0 scale per block of 32 (moe_quantize_mx); only moe_forward_mx takes
 * it. */
typedef enum {
  MOE_DTYPE_F32 = 0,
  MOE_DTYPE_BF16 = 1,
  MOE_DTYPE_E4M3 = 2,
  MOE_DTYPE_MXFP8 = 3
} moe_dtype;

/* Token-tile choice of the grouped GEMMs. AUTO: a batch of T <= 64 tokens
 * uses 32-token tiles (its rows gathered inside the GEMM's loads); larger
 * batches use tiles of up to 256 tokens on pairs of SMs, all experts in one
 * launch, heaviest first, each tile loading only as many token rows as it
 * holds. DECODE, MEDIUM and PREFILL force 32-, 128- or 256-token tiles. */
typedef enum {
  MOE_TILE_AUTO = 0,
  MOE_TILE_DECODE = 1,
  MOE_TILE_PREFILL = 2,
  MOE_TILE_MEDIUM = 3
} moe_tile;

/* Test hooks (moe_problem.flags). Never set in production. */
#define MOE_FLAG_TEST_SKIP_SIGNAL 0x1u /* the GEMM producer withholds its first load
                                          signal, so the consumer's bounded wait runs
                                          out and reports MOE_ERR_TIMEOUT */

typedef struct {
  int64_t T;         /* tokens */
  int64_t H;         /* hidden size */
  int64_t E;         /* routed experts */
  int64_t k;         /* experts per token */
  int64_t I;         /* routed expert intermediate size */
  int64_t I_shared;  /* shared expert intermediate size; 0 = no shared expert */
  int32_t renorm;    /* 1: renormalise the gate weights over the chosen k */
  int32_t dtype;     /* moe_dtype */
  int32_t tile;      /* moe_tile */
  uint32_t flags;    /* MOE_FLAG_* test hooks; 0 in production */
  uint32_t wait_limit_us; /* bound on every device-side wait; 0 = 1 s */
  int32_t out_f32;   /* nonzero: y is written as fp32 even when dtype is bf16 (the
                        sum of the slots before its one rounding to bf16) */
  int32_t n_group;   /* <= 1: plain top-k routing. > 1: group-limited routing (see
                        moe_route_grouped); E % n_group == 0, n_group <= 32 */
  int32_t topk_group; /* groups kept per token when n_group > 1: 1 <= topk_group <=
                         n_group and k <= topk_group * (E / n_group) */
} moe_problem;

/* Bytes of workspace every call below needs for problem `pb`. */
moe_status moe_workspace_size(const moe_problem* pb, size_t* bytes);

/* Step a1, router logits: logits[t][e] = sum_h x[t][h] W_router[e][h]
 * (+ router_bias[e]), fp32 accumulation (the "Gate" at the end of stage 2 in
 * the DeepSeek page's five-stage layer breakdown): bf16 problems on the tensor
 * cores (bf16 products are exact in fp32), fp32 problems on the CUDA cores.
 * router_bias: fp32 [E] or NULL. logits: fp32 [T][E]. */
moe_status moe_router_logits(const moe_problem* pb, const void* x, const void* W_router,
                             const float* router_bias, float* logits, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Step a2, routing (DeepSeek page, "MoE Router"): per token the k largest
 * logits in descending order, lower expert index first among equal logits,
 * and their softmax gate weights (renorm as above). One warp per token.
 * logits fp32 [T][E] -> topk_ids int32 [T][k], topk_w fp32 [T][k]. */
moe_status moe_route(const float* logits, int64_t T, int64_t E, int64_t k, int renorm,
                     int32_t* topk_ids, float* topk_w, void* stream);

/* Step a2, group-limited form (DeepSeek page, "MoE Router": the Mixtral router
 * is the DeepSeek router whose top-K group is the group of all experts). The E
 * experts form n_group contiguous groups of E / n_group. Per token: a group's
 * score is its largest logit; the topk_group groups with the largest scores
 * are kept (lower group index first among equals); then the k largest logits
 * of the kept experts, as moe_route. Gate weights as moe_route, from the
 * unmasked logits (renorm = 0: the softmax over all E). n_group <= 1 is
 * moe_route. Requires E % n_group == 0, n_group <= 32, 1 <= topk_group <=
 * n_group and k <= topk_group * (E / n_group); otherwise MOE_ERR_INVALID_ARG. */
moe_status moe_route_grouped(const float* logits, int64_t T, int64_t E, int64_t k, int renorm,
                             int64_t n_group, int64_t topk_group, int32_t* topk_ids,
                             float* topk_w, void* stream);

/* Step a3, permutation ("CuTeDSL at Perplexity", "Local" dispatch: count the
 * tokens of each expert, give every token a unique index in its expert's
 * list). A stable counting sort of the slots s = t*k + r by expert:
 *   expert_offsets int32 [E+2]: [0..E] exclusive prefix of the per-expert
 *     counts; [E+1] = [E] + (has_shared ? T : 0) closes the shared segment,
 *     whose position T*k + t holds token t;
 *   gather_idx int32 [T*k]: gather_idx[p] = slot at position p (ascending slot
 *     within each expert);
 *   slot_pos int32 [T*k]: slot_pos[s] = position of slot s.
 * No padded buffer is produced. Needs moe_workspace_size() of a problem with
 * these T, E, k (beyond 4096 slots the work is split over CTAs that exchange
 * per-chunk counts through the workspace). Out-of-range ids set
 * MOE_ERR_DEVICE_CHECK in the status. */
moe_status moe_permute(const int32_t* topk_ids, int64_t T, int64_t E, int64_t k,
                       int has_shared, int32_t* expert_offsets, int32_t* gather_idx,
                       int32_t* slot_pos, void* workspace, size_t workspace_bytes,
                       void* stream);

/* Step a4, grouped gate/up GEMM with fused SwiGLU (DeepSeek page "GroupGEMM";
 * Qwen3.5/TPU write-up 4.2.1-4.2.2). expert_offsets, gather_idx and slot_pos
 * are moe_permute's outputs. For every routed position p of expert e
 * (token t = gather_idx[p] / k):
 *   h[p][i] = silu(x[t] . W_gate[e][i]) * (x[t] . W_up[e][i])
 * and, when I_shared > 0, h_shared[t][i] likewise with Ws_gate, Ws_up.
 * Decode-sized token tiles gather the rows of x inside the GEMM's own loads;
 * prefill-sized tiles first copy the routed rows into expert order, unpadded,
 * in the workspace (the dispatch copy of "CuTeDSL at Perplexity", "Local") and
 * load them as whole tiles. Needs moe_workspace_size(pb) bytes of workspace.
 * h: [T*k][I], h_shared: [T][I_shared] (NULL iff I_shared == 0), in the dtype;
 * fp32 accumulation, one rounding to the dtype. */
moe_status moe_grouped_swiglu_gemm(const moe_problem* pb, const void* x,
                                   const int32_t* expert_offsets, const int32_t* gather_idx,
                                   const int32_t* slot_pos, const void* W_gate, const void* W_up,
                                   const void* Ws_gate, const void* Ws_up, void* h,
                                   void* h_shared, void* workspace, size_t workspace_bytes,
                                   void* stream);

/* Step a5 (+a6), down projection and gate-weighted combine (DeepSeek page
 * "Expert Parallelism": weighted sum of the routed outputs plus the shared
 * expert; "CuTeDSL at Perplexity" "Local" combine):
 *   y[t] = sum_r topk_w[t*k+r] * (W_down[e] h[p]) + W_sdown h_shared[t]
 * with p = slot_pos[t*k+r] found through gather_idx. The k products per token
 * are written in fp32 to a slot buffer in the workspace and summed in rank
 * order (then the shared term) by one reduction kernel. y: [T][H] in the
 * dtype, or fp32 when pb->out_f32 is set. */
moe_status moe_down_combine(const moe_problem* pb, const void* h, const void* h_shared,
                            const int32_t* expert_offsets, const int32_t* gather_idx,
                            const float* topk_w, const void* W_down, const void* Ws_down,
                            void* y, void* workspace, size_t workspace_bytes, void* stream);

/* The whole layer: a1 .. a5 (+a6) on `stream`, intermediates in `workspace`.
 * Ws_* are NULL iff pb->I_shared == 0; router_bias may be NULL. */
moe_status moe_forward(const moe_problem* pb, const void* x, const void* W_router,
                       const float* router_bias, const void* W_gate, const void* W_up,
                       const void* W_down, const void* Ws_gate, const void* Ws_up,
                       const void* Ws_down, void* y, void* workspace,
                       size_t workspace_bytes, void* stream);

/* The whole layer (a1 .. a5, a6) as ONE kernel launch, for decode-sized
 * batches: the single-launch decode path ("Lower latency and higher throughput
 * with multi-node DeepSeek deployment", its CUDA-Graph paragraph: persistent
 * kernels that read the per-expert counts on the device; "CuTeDSL at
 * Perplexity": small-batch dispatch inside the kernel that moves the data).
 * Same arguments, layouts, workspace and results as moe_forward: routing ids
 * and the permutation are the same function of the logits; the logits are fp32
 * sums of the same products in another order (one warp per (token, expert),
 * lane-sequential then a fixed butterfly), and y the same computation. One
 * cooperative persistent kernel with one CTA per SM runs: each token's logits
 * and top-k on its own CTA; a grid barrier; the permutation; the gate/up GEMM;
 * the down GEMM, whose units start on an expert as soon as all of that
 * expert's gate/up units are stored (no kernel boundary between the GEMMs); a
 * second grid barrier; the combine. Every cross-CTA wait is bounded by
 * wait_limit_us and reports MOE_ERR_TIMEOUT in the device status.
 * Takes problems that use the 32-token decode tiles (tile AUTO with T <= 64,
 * or DECODE) with dtype bf16 or fp32, T at most the SM count, and whose shared
 * memory fits one CTA per SM (E and T*k not too large); returns
 * MOE_ERR_UNSUPPORTED otherwise, or on a device without cooperative launch.
 * Enqueues a clear of the workspace header (status word and barrier counter)
 * and the one kernel on `stream`. */
moe_status moe_forward_single_launch(const moe_problem* pb, const void* x, const void* W_router,
                                     const float* router_bias, const void* W_gate,
                                     const void* W_up, const void* W_down, const void* Ws_gate,
                                     const void* Ws_up, const void* Ws_down, void* y,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* moe_down_combine without a workspace, for callers that cannot allocate
 * device memory (a host that passes the layer only its inputs and outputs, a
 * plugin not allowed to call cudaMalloc, a fixed memory budget). It computes
 * what moe_down_combine computes, with the same arguments minus the
 * workspace; its scratch (status word + fp32 slot buffer) is one static
 * device array of 16 MiB + 256 bytes inside this library, which every GPU that
 * loads the library holds until the process exits. There is no counterpart on
 * the pages: this is a deployment convenience only.
 *  - Size limit: T * (k + (I_shared > 0)) * H * 4 bytes must not exceed 16 MiB
 *    (e.g. T = 128 decode tokens at H = 4096, k = 8); larger problems return
 *    MOE_ERR_WORKSPACE before any launch.
 *  - Allocates nothing: no cudaMalloc/cudaFree or allocating library call.
 *    The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any
 *    stream capture.
 *  - All calls share the one array: calls that overlap on the GPU (different
 *    streams or threads, same device) race on it and must be serialised by
 *    the caller. The status word is cleared at the start of every call.
 *  - device_status: NULL, or a HOST pointer; when given, the call waits for
 *    `stream` and stores the device status word (MOE_OK, MOE_ERR_TIMEOUT...).
 */
moe_status moe_down_combine_noalloc(const moe_problem* pb, const void* h, const void* h_shared,
                                    const int32_t* expert_offsets, const int32_t* gather_idx,
                                    const float* topk_w, const void* W_down,
                                    const void* Ws_down, void* y, void* stream,
                                    moe_status* device_status);

/* Byte offsets of moe_forward's intermediates inside the workspace (for
 * inspection by tests): logits, topk_ids, topk_w, expert_offsets, gather_idx,
 * slot_pos, h, h_shared. Each is -1 when absent. MXFP8 problems that run the
 * decode-sized kernels (moe_forward_mx) store h and h_shared as E4M3 codes
 * with E8M0 scale rows (moe_mx_scale_cols(I) and (I_shared) bytes per row) at
 * h_scales and h_shared_scales; otherwise those two are -1 and h holds the
 * layer's activation values (bf16 or fp32). */
typedef struct {
  int64_t logits, topk_ids, topk_w, expert_offsets, gather_idx, slot_pos, h, h_shared;
  int64_t h_scales, h_shared_scales;
} moe_workspace_layout;
moe_status moe_get_workspace_layout(const moe_problem* pb, moe_workspace_layout* out);

/* FP8 expert weights ("Hosting Qwen on Blackwell": Qwen3-235B served with FP8
 * microscaled weights converted statically). A matrix is stored as E4M3 codes
 * (OCP 8-bit floating point: 4 exponent bits, bias 7, 3 mantissa bits, largest
 * finite 448, no infinities) with one power-of-two scale per row:
 *   e = the smallest integer with max_i |v_i| <= 448 * 2^e, e >= -126 (e = 0
 *       for a row of zeros); scale = 2^e; q_i = E4M3(v_i / 2^e), nearest even.
 * Scaling by powers of two never rounds, so a value is q * scale and a dot
 * product of two rows is scale_a * scale_b * sum(q_a * q_b).
 * src [rows][cols] bf16 or fp32 (src_dtype), cols a multiple of 16 -> q uint8
 * [rows][cols], scale fp32 [rows]. Device pointers, 16-byte aligned. */
moe_status moe_quantize_rows_e4m3(const void* src, int32_t src_dtype, int64_t rows,
                                  int64_t cols, uint8_t* q, float* scale, void* stream);

/* The layer with E4M3 expert weights: pb->dtype = MOE_DTYPE_E4M3; x, W_router
 * and y are bf16 (y fp32 with out_f32); routing and permutation as moe_forward.
 * Weights are the outputs of moe_quantize_rows_e4m3 over the bf16/fp32 matrices
 * viewed as rows: Wq_gate, Wq_up [E*I][H] with s_gate, s_up [E*I]; Wq_down
 * [E*H][I] with s_down [E*H]; shared Wsq_gate, Wsq_up [I_s][H] with ss_gate,
 * ss_up [I_s]; Wsq_down [H][I_s] with ss_down [H] (all NULL iff I_shared == 0).
 * Per forward pass each token row of x is quantized the same way; the gated
 * GEMM accumulates code products in fp32 and applies both scales, then
 * h = bf16(silu(g) * u); each h row is quantized; the down GEMM applies its
 * scales and the gate weight; the combine is moe_forward's. Requires I and
 * I_shared multiples of 128. Workspace: moe_workspace_size(pb). */
moe_status moe_forward_fp8(const moe_problem* pb, const void* x, const void* W_router,
                           const float* router_bias, const uint8_t* Wq_gate, const float* s_gate,
                           const uint8_t* Wq_up, const float* s_up, const uint8_t* Wq_down,
                           const float* s_down, const uint8_t* Wsq_gate, const float* ss_gate,
                           const uint8_t* Wsq_up, const float* ss_up, const uint8_t* Wsq_down,
                           const float* ss_down, void* y, void* workspace,
                           size_t workspace_bytes, void* stream);

/* MXFP8 expert weights (the MXFP8 serving of Qwen3-235B in "Hosting Qwen on
 * Blackwell", quantization section; the 32-element absolute maxima of "CuTeDSL
 * at Perplexity", Blackwell quantization paragraph). A row of `cols` elements
 * (cols a multiple of 32) is cut into blocks of 32 consecutive elements; per
 * block, with amax its largest magnitude:
 *   e = floor(log2(amax)) - 8, held at -127 from below; e = -127 for zeros;
 *   scale byte = e + 127 (E8M0: the scale is 2^(byte - 127));
 *   codes = E4M3(v / 2^e), nearest even, clamped to +-448.
 * Scale rows are moe_mx_scale_cols(cols) = 16 * ceil(cols / 512) bytes: the
 * row's cols / 32 scale bytes, then zeros.
 * src [rows][cols] bf16 or fp32 (src_dtype) -> q uint8 [rows][cols], scales
 * uint8 [rows][moe_mx_scale_cols(cols)]. Device pointers, 16-byte aligned. */
int64_t moe_mx_scale_cols(int64_t cols);
moe_status moe_quantize_mx(const void* src, int32_t src_dtype, int64_t rows, int64_t cols,
                           uint8_t* q, uint8_t* scales, void* stream);

/* The layer with MXFP8 expert weights: pb->dtype = MOE_DTYPE_MXFP8; x,
 * W_router and y are bf16 (y fp32 with out_f32); routing and permutation as
 * moe_forward (on x itself). Weights are moe_quantize_mx of the matrices viewed
 * as rows over their contraction axis: Wq_gate, Wq_up [E*I][H] with s_gate,
 * s_up [E*I][moe_mx_scale_cols(H)]; Wq_down [E*H][I] with s_down
 * [E*H][moe_mx_scale_cols(I)]; the shared expert's Wsq_gate, Wsq_up [I_s][H],
 * Wsq_down [H][I_s] with their scales (all NULL iff I_shared == 0).
 * Per forward pass each token row of x is quantized the same way (blocks of
 * 32 along H); both GEMMs multiply the bf16 values of the MXFP8 operands (a
 * code times its block scale is a bf16 value, exactly for scales of 2^-117 and
 * above) with fp32 accumulation; h = silu(g) * u is quantized from fp32 per
 * block of 32 along I and stored as its bf16 values; the down GEMM applies the
 * gate weight; the combine is moe_forward's. Requires I and I_shared multiples
 * of 128 and H, I, I_shared <= 8192 (else MOE_ERR_UNSUPPORTED), and problems
 * whose tiles fit the device's shared memory (MOE_ERR_UNSUPPORTED otherwise).
 * Workspace: moe_workspace_size(pb). */
moe_status moe_forward_mx(const moe_problem* pb, const void* x, const void* W_router,
                          const float* router_bias, const uint8_t* Wq_gate, const uint8_t* s_gate,
                          const uint8_t* Wq_up, const uint8_t* s_up, const uint8_t* Wq_down,
                          const uint8_t* s_down, const uint8_t* Wsq_gate, const uint8_t* ss_gate,
                          const uint8_t* Wsq_up, const uint8_t* ss_up, const uint8_t* Wsq_down,
                          const uint8_t* ss_down, void* y, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Synchronises `stream`, then copies the device status word into *out. */
moe_status moe_get_device_status(const void* workspace, void* stream, moe_status* out);

/* Enqueues a clear of the device status word on `stream`. */
moe_status moe_reset_device_status(void* workspace, void* stream);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_API_H_ */
