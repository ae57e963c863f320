/*
 * moefp8.h -- C ABI of libmoefp8.so, the FP8-quantized MoE expert FFN on
 * GB300 (sm_103a).
 *
 * The path, in order (forward):
 *   1. moe_quantize_rows      bf16 activations -> e4m3 codes + fp32 scales
 *   2. moe_ragged_sort        stable sort of the (token, expert) pairs by
 *                             expert; gathers the quantised rows and scales
 *   3. gmm_fp8                grouped matmul with [wi_0 | wi_1]
 *   4. moe_swiglu_quant       h = silu(a0) * a1, requantised like step 1
 *   5. gmm_fp8                grouped matmul with wo
 *   6. ragged_gather_reduce   undo the sort, sum the top-k rows weighted by
 *                             the router probabilities
 * and, for the weight-gradient pass, tgmm_fp8 plus the helpers
 * moe_gather_scale_quant, moe_swiglu_bwd_quant and moe_quantize_group_cols.
 *
 * Sources (MaxText pull-request pages):
 *   [Q-EP]   "Quantize activations before EP all gather" (PR #4812).
 *   [Q-GMM]  "Support quantization for tokamax gmm v2" (PR #4451).
 *   [Q-FUSE] "Keep qwix out of tpu-inference's fused MoE kernel and
 *            pre-quantize weights" (PR #5136).
 *
 * Conventions, for every entry point unless stated otherwise:
 *   - Every pointer is a DEVICE pointer owned by the caller; the library
 *     never frees or retains it.  Pointers must be 16-byte aligned.
 *   - bf16 tensors are passed as uint16_t bit patterns; e4m3 tensors
 *     ("float8_e4m3fn") as uint8_t codes; scales are IEEE fp32.
 *   - Matrices are row-major and dense (row pitch = columns).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and returns before the GPU work finishes.
 *   - The library allocates no device memory.  Kernels that need scratch
 *     memory take a caller-provided workspace whose size a *_workspace_bytes
 *     function reports.
 *   - On a non-OK status nothing was launched, unless the status is
 *     MOE_ERR_CUDA (a launch failed part way).  Outputs are undefined after
 *     any error.
 *   - Data-dependent problems found on the GPU (an expert id outside [0, E),
 *     group sizes that do not add up, a bounded wait that ran out) set a
 *     sticky device error word instead of faulting; the affected kernel
 *     stops early.  Read and clear it with moe_get_device_error.
 */
#ifndef MOEFP8_H_
#define MOEFP8_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* moe_stream_t; /* a cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, bad mode */
  MOE_ERR_UNSUPPORTED = 2, /* shape or mode not built, or device is not sm_103 */
  MOE_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE = 4       /* the device error word was non-zero */
} moe_status;

/* Scale modes.  The shape of a scale tensor follows from the mode:
 *   MOE_SCALE_PER_ROW           [rows]            one scale per row (per token;
 *                                                 for weights: per output channel)
 *   MOE_SCALE_PER_ROW_BLOCK128  [rows, cols/128]  per row and per 128 columns
 *                                                 (weights: see gmm_fp8)
 *   MOE_SCALE_PER_TENSOR        [1]               one fixed scale (static scheme)
 *   MOE_SCALE_PER_GROUP_COL     [E_local, cols]   one scale per (expert, column),
 *                                                 for tgmm operands only */
typedef enum {
  MOE_SCALE_PER_ROW = 0,
  MOE_SCALE_PER_ROW_BLOCK128 = 1,
  MOE_SCALE_PER_TENSOR = 2,
  MOE_SCALE_PER_GROUP_COL = 3
} moe_scale_mode;

/* Device error word bits. */
#define MOE_DEVERR_BAD_EXPERT_ID 0x1u /* moe_ragged_sort: id outside [0, E) */
#define MOE_DEVERR_GROUP_SIZES 0x2u   /* gmm/tgmm: negative size or sum != M */
#define MOE_DEVERR_TIMEOUT 0x4u       /* a bounded wait in a tcgen05 kernel ran out */
#define MOE_DEVERR_TMEM 0x8u          /* tensor-memory allocation returned no columns */
#define MOE_DEVERR_BAD_POSITION 0x10u /* ragged_gather_reduce: a pos entry outside [0, T*k) */

const char* moe_status_string(moe_status s);

/* Synchronises `stream`, stores the device error word of the current device
 * in *code (0 = none) and clears it.  Returns MOE_ERR_DEVICE when *code != 0,
 * MOE_ERR_CUDA when synchronisation failed, else MOE_OK. */
moe_status moe_get_device_error(moe_stream_t stream, int* code);

/* Number of streaming multiprocessors the persistent kernels size their grid
 * by (the current device's SM count); 0 on error. */
int moe_num_sms(void);

/* Test hook for the failure path of the tensor-core kernels: while
 * limit_ns != 0, the epilogue warps of every following gmm_fp8 launch first
 * wait on a barrier that nothing arrives on, bounded by limit_ns.  The wait
 * runs out, the kernel stops its producer and MMA issuer, lets their issued
 * loads and MMAs finish, frees its tensor memory, returns and sets
 * MOE_DEVERR_TIMEOUT; the output is undefined.  0 restores normal operation.
 * Process-wide; not for production use. */
void moe_test_stall_epilogue(uint64_t limit_ns);

/* ------------------------------------------------------------------------
 * Step 1 -- activation quantisation ([Q-EP] description: quantise before the
 * all-gather and the activation sort; [Q-GMM] review reply: fp8_dynamic uses
 * absmax scales, fp8_static_wa fixed activation scales).
 *
 *   s = fp32(amax / 448)   (s = 1 when amax = 0)
 *   q = e4m3(fp32(x / s))  round to nearest even, |v| > 448 saturates, the
 *                          sign of zero is kept.
 * x: bf16 [rows, cols].  q: e4m3 [rows, cols].
 * mode PER_ROW: scale [rows]; PER_ROW_BLOCK128: scale [rows, cols/128];
 * PER_TENSOR: static_scale (device, [1]) is used and `scale` is not written
 * (may be NULL).  cols % 16 == 0 (a last block narrower than 128 columns
 * takes its own scale); cols <= 32768; rows < 2^31.
 */
moe_status moe_quantize_rows(const uint16_t* x, int64_t rows, int64_t cols, moe_scale_mode mode,
                             const float* static_scale, uint8_t* q, float* scale, moe_stream_t stream);

/* Weight pre-quantisation ([Q-FUSE]: weights pre-quantised to float8_e4m3fn
 * with [E, blocks, 1, N] scales).  w: bf16 [E, N, K] (output channel major,
 * the contracted dimension K contiguous).  Each (e, n) row is quantised as in
 * moe_quantize_rows.  Scale layouts: PER_ROW (per channel) [E, N];
 * PER_ROW_BLOCK128 (blockwise) [E, K/128, N], the pages' [E, blocks, 1, N];
 * PER_TENSOR uses static_scale.  K % 16 == 0 (% 128 for blockwise). */
moe_status moe_quantize_weights(const uint16_t* w, int64_t E, int64_t N, int64_t K, moe_scale_mode mode,
                                const float* static_scale, uint8_t* q, float* scale, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Step 2 -- ragged sort by routed expert, plus the gather of quantised rows
 * and row scales ([Q-EP] review threads on ragged_sort / ragged_gather: the
 * scale rows are gathered only when the scale's leading dimension is the
 * token dimension).
 *
 * topk_ids: int32 [T, k]; flat pair i = t*k + j.  Stable counting sort by
 * expert id, then by i.  Outputs:
 *   sorted_src    int32 [T*k]   flat pair index at sorted position r
 *   pos           int32 [T*k]   inverse: sorted position of pair i
 *   group_sizes   int32 [E]
 *   group_offsets int32 [E+1]   exclusive prefix sum of group_sizes
 *   xs_q          e4m3 [T*k, D] xs_q[r] = x_q[sorted_src[r] / k]
 *   xs_scale      PER_ROW: [T*k]; PER_ROW_BLOCK128: [T*k, D/128];
 *                 PER_TENSOR: not written (may be NULL)
 * workspace: device scratch of moe_ragged_sort_workspace_bytes(T, k, E)
 * bytes (its contents need not be initialised).  An id outside [0, E) sets
 * MOE_DEVERR_BAD_EXPERT_ID.  D % 16 == 0; 1 <= k <= 32; E <= 1024;
 * T*k < 2^31.
 */
size_t moe_ragged_sort_workspace_bytes(int64_t T, int k, int E);
moe_status moe_ragged_sort(const int32_t* topk_ids, int64_t T, int k, int E, const uint8_t* x_q,
                           const float* x_scale, int64_t D, moe_scale_mode mode, int32_t* sorted_src, int32_t* pos,
                           int32_t* group_sizes, int32_t* group_offsets, uint8_t* xs_q, float* xs_scale,
                           void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* moe_quantize_sort -- steps 1 and 2 in one call: the sort indices as in
 * moe_ragged_sort, and the activation quantisation of moe_quantize_rows
 * (same scale rule and modes) fused into the gather, so the token-order codes
 * never go to memory: each token row of x is quantised once and its codes and
 * scales are written to its k sorted rows.  Row by row, gather(quantize(x)) is
 * quantize(gather(x)) ("Quantize activations before EP all gather": the
 * quantisation moves ahead of the gather at no cost), so xs_q and xs_scale are
 * bit-identical to moe_quantize_rows followed by moe_ragged_sort.
 *   x bf16 [T, D]; static_scale [1] for PER_TENSOR (else unused);
 *   xs_scale [T*k] (PER_ROW) or [T*k, D/128] (PER_ROW_BLOCK128), 16-byte
 *   aligned; every other argument as moe_ragged_sort (same workspace size).
 * D % 16 == 0, D <= 32768.  Invalid ids raise MOE_DEVERR_BAD_EXPERT_ID. */
moe_status moe_quantize_sort(const uint16_t* x, const int32_t* topk_ids, int64_t T, int k, int E, int64_t D,
                             moe_scale_mode mode, const float* static_scale, int32_t* sorted_src, int32_t* pos,
                             int32_t* group_sizes, int32_t* group_offsets, uint8_t* xs_q, float* xs_scale,
                             void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* moe_ragged_sort_noalloc -- moe_ragged_sort for callers that cannot
 * allocate device memory.  The pages have no counterpart: it exists for
 * hosts that own every byte of device memory themselves (an inference engine
 * whose pool has already claimed the free HBM, a plugin interface that hands
 * out no allocator) and for latency-critical loops where cudaMalloc, which
 * may synchronise the device, is not allowed.  Arguments and results are
 * those of moe_ragged_sort without the workspace.
 *
 * The scratch is a fixed device array of MOE_RAGGED_SORT_NOALLOC_SCRATCH_BYTES
 * (1 MiB) inside the library; every GPU that loads the library holds it
 * until the process exits.  Problems for which
 * moe_ragged_sort_workspace_bytes(T, k, E) exceeds it -- with E = 256, more
 * than 2^21 (token, expert) pairs -- are rejected with MOE_ERR_INVALID_ARG
 * before anything is launched.  The first call on a device looks up the
 * array's device address (once per device, with that device current); make
 * that first call before any stream capture.  All calls on a device share
 * the one array: calls that overlap on the GPU (on different streams, or from
 * different host threads) race and corrupt each other's results.  Each call
 * writes every count it reads, so nothing carries over between calls.  No
 * device memory is allocated or freed. */
#define MOE_RAGGED_SORT_NOALLOC_SCRATCH_BYTES (1u << 20)
moe_status moe_ragged_sort_noalloc(const int32_t* topk_ids, int64_t T, int k, int E, const uint8_t* x_q,
                                   const float* x_scale, int64_t D, moe_scale_mode mode, int32_t* sorted_src,
                                   int32_t* pos, int32_t* group_sizes, int32_t* group_offsets, uint8_t* xs_q,
                                   float* xs_scale, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Steps 3 and 5 -- grouped matmul ([Q-EP] review on gmm_v2: gmm(lhs_q,
 * rhs_q, group_sizes, rhs_scale, group_offset) on already-quantised lhs, the
 * lhs scale multiplying the output; bf16 output for fp8 operands; [Q-FUSE]:
 * fp32 accumulation).
 *
 *   out[m, n] = sum_k deq(lhs)[m, k] * deq(rhs)[g(m) - group_offset, n, k]
 *
 * g(m) is the group holding row m (groups are consecutive row ranges of
 * sizes group_sizes[0..E)).  Only groups [group_offset, group_offset +
 * E_local) are computed; all other rows of out are written as zero.
 *   lhs_q     e4m3 [M, K];  lhs_scale: PER_ROW [M], PER_ROW_BLOCK128
 *             [M, K/128] or PER_TENSOR [1]
 *   rhs_q     e4m3 [E_local, N, K] (K contiguous);  rhs_scale: PER_ROW (per
 *             channel) [E_local, N], PER_ROW_BLOCK128 (blockwise)
 *             [E_local, K/128, N], or PER_TENSOR [1]
 *   out       bf16 [M, N], fp32 accumulation on the tensor cores; with a
 *             blockwise operand each 128-wide K block is scaled and summed in
 *             fp32 registers.
 * Requires K % 16 == 0 (K % 128 == 0 when either side is blockwise),
 * N % 16 == 0, sum(group_sizes) == M (else MOE_DEVERR_GROUP_SIZES), E <= 1024.
 * Returns MOE_ERR_UNSUPPORTED on a device other than sm_103.
 */
moe_status gmm_fp8(const uint8_t* lhs_q, const float* lhs_scale, moe_scale_mode lhs_mode, const uint8_t* rhs_q,
                   const float* rhs_scale, moe_scale_mode rhs_mode, const int32_t* group_sizes, int E,
                   int group_offset, int E_local, int64_t M, int64_t K, int64_t N, uint16_t* out,
                   moe_stream_t stream);

/* gmm_fp8_ksplit -- grouped matmul whose K range is two segments, each with
 * one static weight scale: the backward's input gradient
 * dXs = dA0 W0^T + dA1 W1^T as one contraction over [dA0 | dA1] (K = 2F,
 * K_split = F) with rhs = [W0 | W1]^T, the static scales s0 of wi_0 and s1 of
 * wi_1 ("Support quantization for tokamax gmm v2": fp8_static_wa):
 *   out[m, n] = bf16( (s0 * sum_{k < K_split} a[m,k] w[g,n,k]
 *                    + s1 * sum_{k >= K_split} a[m,k] w[g,n,k]) * s_a[m] )
 * Both sums are fp32 on the tensor cores, in two accumulators that meet in the
 * epilogue (no per-128 promotion).  lhs_mode PER_ROW [M] or PER_TENSOR [1];
 * rhs_scale2 = {s0, s1} (device, 2 floats); rhs_q [E_local, N, K].
 * K_split % 128 == 0, 0 <= K_split <= K; otherwise as gmm_fp8. */
moe_status gmm_fp8_ksplit(const uint8_t* lhs_q, const float* lhs_scale, moe_scale_mode lhs_mode,
                          const uint8_t* rhs_q, const float* rhs_scale2, int64_t K_split,
                          const int32_t* group_sizes, int E, int group_offset, int E_local, int64_t M, int64_t K,
                          int64_t N, uint16_t* out, moe_stream_t stream);

/* gmm_fp8_swiglu -- steps 3 and 4 in one pass: the [wi_0 | wi_1] grouped
 * matmul with SwiGLU and the requantisation of h in its epilogue, so the
 * [M, 2F] bf16 product a never goes to memory.  Bit-identical to gmm_fp8
 * (rhs = [wi_0 | wi_1], N = 2F) followed by moe_swiglu_quant: every output tile
 * holds matching wi_0 and wi_1 channels, a0 and a1 are rounded to bf16 exactly
 * as gmm_fp8 stores them, and h = bf16(silu(a0) a1) is computed the same way.
 *   lhs_q e4m3 [M, K], lhs_scale PER_ROW [M], PER_ROW_BLOCK128 [M, K/128] or
 *         PER_TENSOR [1]
 *   rhs_q e4m3 [E_local, 2F, K] (wi_0 channels, then wi_1 channels),
 *         rhs_scale PER_ROW (per channel) [E_local, 2F], PER_ROW_BLOCK128
 *         (blockwise) [E_local, K/128, 2F] or PER_TENSOR [1]
 *   h_mode PER_ROW: h_scale [M]; `h` is bf16 [M, F] scratch that receives h
 *          (the row's scale needs all of its F columns first)
 *   h_mode PER_ROW_BLOCK128: h_scale [M, F/128], fully fused (h may be NULL):
 *          a 128-column h block is one output tile
 *   h_mode PER_TENSOR: h_static_scale [1], fully fused (h may be NULL)
 *   h_q   e4m3 [M, F]
 *   a_out optional bf16 [M, 2F]: also store a = [a0 | a1] (for a backward pass)
 * With a blockwise operand scale ("Keep qwix out of tpu-inference's fused MoE
 * kernel and pre-quantize weights": [E, blocks, 1, N] weight scales) each
 * 128-wide K block is scaled and summed in fp32 registers, as in gmm_fp8.
 * Rows outside groups [group_offset, group_offset + E_local) get zero codes
 * and scale 1; a_out and h are not written there.  F % 128 == 0, K % 16 == 0
 * (K % 128 == 0 with a blockwise scale), sum(group_sizes) == M, E <= 1024.
 * MOE_ERR_UNSUPPORTED off sm_103. */
moe_status gmm_fp8_swiglu(const uint8_t* lhs_q, const float* lhs_scale, moe_scale_mode lhs_mode,
                          const uint8_t* rhs_q, const float* rhs_scale, moe_scale_mode rhs_mode,
                          const int32_t* group_sizes, int E, int group_offset, int E_local, int64_t M, int64_t K,
                          int64_t F, moe_scale_mode h_mode, const float* h_static_scale, uint16_t* a_out,
                          uint16_t* h, uint8_t* h_q, float* h_scale, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Step 4 -- SwiGLU and requantisation.  a = [a0 | a1], bf16 [R, 2F] (the
 * wi_0 | wi_1 gmm output).  h = bf16(silu(a0) * a1) in fp32 with
 * silu(z) = z / (1 + e^-z); h is quantised exactly as moe_quantize_rows does
 * (same modes and scale shapes, cols = F).  F % 16 == 0, F <= 32768.
 */
moe_status moe_swiglu_quant(const uint16_t* a, int64_t R, int64_t F, moe_scale_mode mode,
                            const float* static_scale, uint8_t* h_q, float* h_scale, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Step 6 -- ragged gather-reduce ([Q-EP]: ragged_gather_reduce un-permutes
 * the expert outputs and sums the top-k rows of each token):
 *   out[t, :] = bf16( sum_{j<k} weights[t, j] * rows[pos[t*k + j], :] )
 * fp32 accumulation in ascending j.  rows bf16 [T*k, D]; pos int32 [T*k];
 * weights fp32 [T, k] or NULL (all ones); out bf16 [T, D].  D % 8 == 0;
 * 1 <= k <= 32; T*k < 2^31.  A pos entry outside [0, T*k) contributes
 * nothing to its token's sum and sets MOE_DEVERR_BAD_POSITION.
 */
moe_status ragged_gather_reduce(const uint16_t* rows, const int32_t* pos, const float* weights, int64_t T, int k,
                                int64_t D, uint16_t* out, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Backward helpers ([Q-GMM]: gmm and tgmm gradients, "absmax grad").
 *
 * moe_gather_scale_quant -- adjoint of the combine, fused with per-row
 * quantisation:  dO[r] = bf16(fp32(w[i] * G[i / k])), i = sorted_src[r];
 * then dO_q, dO_scale = per-row quantisation of dO as in moe_quantize_rows.
 * G bf16 [T, D]; w fp32 [T*k] (NULL: ones); dO bf16 [T*k, D]; dO_q e4m3
 * [T*k, D]; dO_scale [T*k].  D % 16 == 0.
 */
moe_status moe_gather_scale_quant(const uint16_t* G, const float* w, const int32_t* sorted_src, int64_t T, int k,
                                  int64_t D, uint16_t* dO, uint8_t* dO_q, float* dO_scale, moe_stream_t stream);

/* moe_swiglu_bwd_quant -- SwiGLU backward in fp32, rounded to bf16, fused
 * with per-row quantisation of the concatenated [dA0 | dA1] row:
 *   sigma = 1/(1 + e^-a0), silu = a0/(1 + e^-a0),
 *   dA0 = (dH * a1) * sigma (1 + a0 (1 - sigma)),   dA1 = dH * silu.
 * dH bf16 [R, F]; a bf16 [R, 2F]; dA bf16 [R, 2F]; dA_q e4m3 [R, 2F];
 * dA_scale [R].  F % 16 == 0, 2F <= 32768. */
moe_status moe_swiglu_bwd_quant(const uint16_t* dH, const uint16_t* a, int64_t R, int64_t F, uint16_t* dA,
                                uint8_t* dA_q, float* dA_scale, moe_stream_t stream);

/* moe_quantize_group_cols -- requantise a gradient with one absmax scale per
 * (expert, column) over that expert's rows, so that both scales of the
 * weight-gradient contraction factor out of the sum over rows.
 * g bf16 [M, N]; q e4m3 [M, N] (rows outside the local groups are not
 * written), or NULL for the scales only (tgmm_fp8_gcq then makes the codes);
 * scale fp32 [E_local, N] (an expert without rows, or an all-zero column,
 * gets 1).  N % 16 == 0, E <= 1024.  `scale` is also used as the running
 * maximum while the kernel runs. */
moe_status moe_quantize_group_cols(const uint16_t* g, int64_t M, int64_t N, const int32_t* group_sizes, int E,
                                   int group_offset, int E_local, uint8_t* q, float* scale, moe_stream_t stream);

/* tgmm_fp8 -- transposed grouped matmul for weight gradients ([Q-GMM]:
 * tgmm for grad_wi_0, grad_wi_1 and grad_wo):
 *   out[e, k, n] = sum_{m in group e} deq(lhs)[m, k] * deq(rhs)[m, n]
 * for local groups e in [0, E_local) (global group group_offset + e).
 *   lhs_q e4m3 [M, K], lhs_scale PER_TENSOR [1] or PER_GROUP_COL [E_local, K]
 *   rhs_q e4m3 [M, N], rhs_scale PER_TENSOR [1] or PER_GROUP_COL [E_local, N]
 *   out   fp32 [E_local, K, N]; an expert without rows gets zeros.
 * workspace: tgmm_fp8_workspace_bytes(M, K, N, E_local) bytes of device
 * scratch (no initialisation needed); it holds both operands transposed, each
 * group padded to 128 rows.  K % 16 == 0, N % 16 == 0, E <= 1024.
 * Returns MOE_ERR_UNSUPPORTED on a device other than sm_103.
 */
size_t tgmm_fp8_workspace_bytes(int64_t M, int64_t K, int64_t N, int E_local);
moe_status tgmm_fp8(const uint8_t* lhs_q, const float* lhs_scale, moe_scale_mode lhs_mode, const uint8_t* rhs_q,
                    const float* rhs_scale, moe_scale_mode rhs_mode, const int32_t* group_sizes, int E,
                    int group_offset, int E_local, int64_t M, int64_t K, int64_t N, float* out, void* workspace,
                    size_t workspace_bytes, moe_stream_t stream);

/* tgmm_fp8_gcq -- tgmm_fp8 whose rhs is given as the bf16 gradient g [M, N]
 * with its finished per-(expert, column) scales (moe_quantize_group_cols with
 * q == NULL): the e4m3 codes of g are made while g is laid out transposed and
 * group-padded in the workspace, so the row-major codes never go to memory.
 * The codes, and so the result, are those of moe_quantize_group_cols followed
 * by tgmm_fp8 with rhs_mode PER_GROUP_COL.  Other arguments as tgmm_fp8. */
moe_status tgmm_fp8_gcq(const uint8_t* lhs_q, const float* lhs_scale, moe_scale_mode lhs_mode, const uint16_t* rhs_g,
                        const float* rhs_scale, const int32_t* group_sizes, int E, int group_offset, int E_local,
                        int64_t M, int64_t K, int64_t N, float* out, void* workspace, size_t workspace_bytes,
                        moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Router ([Q-GMM] table 1 measures the gate kernel's gradient grad_gate-kernel
 * and the state gradient state_grad beside the expert weights' gradients).
 *
 * moe_router_topk -- the gate layer and the routing decision in one call:
 *   logits[t, e] = sum_d x[t, d] w_gate[e, d]   (bf16 operands, fp32
 *                                                accumulation on the tensor cores)
 *   p = softmax over the E logits of the row, in fp32: m = max, e_i =
 *       exp(l_i - m), Z = e_0 + e_1 + ... in ascending i, p_i = e_i / Z
 *   topk_ids[t, :] = the k most probable experts in descending order of p,
 *                    ties to the lower expert index;
 *   topk_w[t, j]   = p[topk_ids[t, j]] (not renormalised).
 * x bf16 [T, D]; w_gate bf16 [E, D]; logits fp32 [T, E] (kept for the
 * backward); topk_ids int32 [T, k]; topk_w fp32 [T, k].  D % 8 == 0,
 * 1 <= E <= 256, 1 <= k <= min(8, E); every row needs a finite logit. */
moe_status moe_router_topk(const uint16_t* x, const uint16_t* w_gate, int64_t T, int64_t D, int E, int k,
                           float* logits, int32_t* topk_ids, float* topk_w, moe_stream_t stream);

/* moe_router_backward -- the router's gradient from the combine's output
 * gradient G (the expert FFN's dY):
 *   dw[t, j]      = <G[t], o[pos[t k + j]]>        fp32 [T, k]
 *   dlogits[t, i] = bf16( p_i (g_i - s) )          bf16 [T, E]
 *                   with p recomputed from logits as in moe_router_topk,
 *                   s = sum_j p[id_j] dw[t, j] (ascending j), g_i = dw[t, j]
 *                   for i = id_j, else 0
 *   grad_gate     = dlogits^T x                    fp32 [E, D] (w_gate's layout)
 *   state_grad    = dlogits w_gate                 bf16 [T, D] (the gradient
 *                                                   reaching x through the router)
 * G bf16 [T, D]; o bf16 [T*k, D] (the expert outputs of the forward);
 * pos int32 [T*k] (moe_ragged_sort); x, w_gate, logits, topk_ids as given to
 * / returned by moe_router_topk.  workspace: moe_router_backward_workspace_bytes
 * bytes (x and w_gate transposed, dlogits padded and transposed).
 * D % 16 == 0, T <= 2^21, 1 <= E <= 256, 1 <= k <= min(8, E). */
size_t moe_router_backward_workspace_bytes(int64_t T, int64_t D, int E);
moe_status moe_router_backward(const uint16_t* G, const uint16_t* o, const int32_t* pos, const uint16_t* x,
                               const uint16_t* w_gate, const float* logits, const int32_t* topk_ids, int64_t T,
                               int64_t D, int E, int k, float* dw, uint16_t* dlogits, float* grad_gate,
                               uint16_t* state_grad, void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* moe_transpose_u8 -- weight layout preparation for the backward pass (run
 * once, outside the FFN): batched byte transpose src [B, R, C] -> dst
 * [B, C, R] of e4m3 codes.  The input-gradient gmm contracts over the
 * weights' output channels, so it reads the weights transposed.  With a
 * per-tensor weight scale the transposed codes are exactly the codes of the
 * transposed weights.  R % 16 == 0, C % 16 == 0. */
moe_status moe_transpose_u8(const uint8_t* src, int64_t B, int64_t R, int64_t C, uint8_t* dst, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * MXFP8 variant of steps 1-5.  It is not a method of the three pages: it is
 * the same path on Blackwell's block-scaled tensor-core format, as defined by
 * the OCP "Microscaling Formats (MX) Specification" v1.0 (MXFP8, E4M3
 * elements).
 *
 * Every 32 consecutive values of a row along the contracted dimension form a
 * block.  A block shares one E8M0 scale 2^X, stored as the byte X + 127:
 *   X = floor(log2(amax)) - 8   clamped to [-127, 127]; X = -127 when amax = 0
 *   q = e4m3(x / 2^X)           round to nearest even, saturating at 448.
 *   (8 is the exponent of 256, the largest power of two in e4m3.)
 * E8M0 tensors are K-block-major: uint8_t [cols/128][rows][4].  The code of
 * (row, 32-column block b) is at ((b / 4) * rows + row) * 4 + b % 4.  So the
 * four codes of a row's 128-column block form one 32-bit word, and for one
 * 128-column block the words of consecutive rows are adjacent: a tile of rows
 * reads its codes for one K step as one contiguous run.  cols is a multiple of
 * 128.
 *
 * The grouped matmuls run tcgen05.mma.kind::mxf8f6f4.block_scale.  The
 * tensor core applies both operands' scales to each 32-wide K block, so
 * accumulation stays in fp32 tensor memory across the whole K loop.
 * ------------------------------------------------------------------------ */

/* Step 1 (MX).  x bf16 [rows, cols] -> q e4m3 [rows, cols], sf E8M0
 * [cols/128][rows][4].  Expert weights w[E, N, K] are passed as rows = E*N,
 * cols = K: their codes are [K/128][E*N][4].  cols % 128 == 0,
 * cols <= 32768, rows < 2^31; x and q 16-byte aligned. */
moe_status moe_quantize_rows_mx(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* q, uint8_t* sf,
                                moe_stream_t stream);

/* Steps 1 + 2 (MX), as moe_quantize_sort: the sort indices, and each token
 * row quantised once with its codes and E8M0 codes written to its k sorted
 * rows.  xs_q [T*k, D], xs_sf [D/128][T*k][4]; workspace as moe_ragged_sort.
 * D % 128 == 0, D <= 32768. */
moe_status moe_quantize_sort_mx(const uint16_t* x, const int32_t* topk_ids, int64_t T, int k, int E, int64_t D,
                                int32_t* sorted_src, int32_t* pos, int32_t* group_sizes, int32_t* group_offsets,
                                uint8_t* xs_q, uint8_t* xs_sf, void* workspace, size_t workspace_bytes,
                                moe_stream_t stream);

/* Steps 3 / 5 (MX).  out[m, n] = bf16( sum_k deq(lhs)[m, k] deq(rhs)[g(m), n, k] )
 * with deq(x)[.., k] = e4m3(x[.., k]) * 2^(sf[.., k/32] - 127).
 *   lhs_q [M, K], lhs_sf [K/128][M][4]; rhs_q [E_local, N, K], rhs_sf
 *   [K/128][E_local * N][4] (row e * N + n); out bf16 [M, N].
 * Groups, group_offset and E_local are as in gmm_fp8: rows outside the
 * local groups are zero.  K % 128 == 0, N % 16 == 0.  Every pointer is
 * 16-byte aligned. */
moe_status gmm_fp8_mx(const uint8_t* lhs_q, const uint8_t* lhs_sf, const uint8_t* rhs_q, const uint8_t* rhs_sf,
                      const int32_t* group_sizes, int E, int group_offset, int E_local, int64_t M, int64_t K,
                      int64_t N, uint16_t* out, moe_stream_t stream);

/* Steps 3 + 4 (MX) in one kernel.  rhs_q [E_local, 2F, K] holds the wi_0
 * rows and then the wi_1 rows of each expert, rhs_sf [K/128][E_local*2F][4].
 * The epilogue:
 *   - rounds a0 and a1 to bf16 as gmm_fp8_mx would store them;
 *   - forms h = bf16(silu(a0) * a1) (the h of moe_swiglu_quant);
 *   - quantises h per 32 columns into h_q [M, F] and h_sf [F/128][M][4].
 * a_out (optional, may be NULL) receives the bf16 [a0 | a1] [M, 2F].
 * Rows outside the local groups get zero codes and E8M0 code 0.
 * K % 128 == 0, F % 128 == 0; every pointer 16-byte aligned. */
moe_status gmm_fp8_mx_swiglu(const uint8_t* lhs_q, const uint8_t* lhs_sf, const uint8_t* rhs_q, const uint8_t* rhs_sf,
                             const int32_t* group_sizes, int E, int group_offset, int E_local, int64_t M, int64_t K,
                             int64_t F, uint16_t* a_out, uint8_t* h_q, uint8_t* h_sf, moe_stream_t stream);

/* Step 4 (MX), unfused: a = [a0 | a1] bf16 [R, 2F] -> h = bf16(silu(a0) a1)
 * quantised per 32 columns: h_q [R, F], h_sf [F/128][R][4].  F % 128 == 0. */
moe_status moe_swiglu_quant_mx(const uint16_t* a, int64_t R, int64_t F, uint8_t* h_q, uint8_t* h_sf,
                               moe_stream_t stream);

/* ------------------------------------------------------------------------
 * int8-weight variant of steps 3 and 5 ([Q-FUSE], "Keep qwix out of
 * tpu-inference's fused MoE kernel and pre-quantize weights", description:
 * the weights are pre-quantised to float8_e4m3fn or int8 with [E, blocks, 1,
 * N] scales).  The activations and h stay e4m3 with their scales, and steps
 * 1, 2, 4 and 6 are unchanged.
 *
 * int8 codes are symmetric absmax:
 *   s = fp32(amax / 127), s = 1 when amax = 0;
 *   q = nearest integer of fp32(x / s), ties to even, limited to [-127, 127].
 * ------------------------------------------------------------------------ */

/* Weights w[E, N, K] bf16 -> int8 codes q[E, N, K] and fp32 scales in the
 * layouts of moe_quantize_weights: PER_ROW (per channel) [E, N];
 * PER_ROW_BLOCK128 (blockwise) [E, K/128, N]; PER_TENSOR uses static_scale.
 * K % 16 == 0 (% 128 for blockwise), K <= 32768; w and q 16-byte aligned. */
moe_status moe_quantize_weights_int8(const uint16_t* w, int64_t E, int64_t N, int64_t K, moe_scale_mode mode,
                                     const float* static_scale, int8_t* q, float* scale, moe_stream_t stream);

/* Steps 3 / 5 with int8 weights:
 *   out[m, n] = bf16( sum_k deq(lhs)[m, k] * q[g(m), n, k] * s_w )
 * with deq(lhs) as in gmm_fp8 (lhs_mode PER_ROW or PER_TENSOR), q the int8
 * code as an integer and s_w its weight scale (rhs_mode PER_ROW [E_local, N],
 * PER_ROW_BLOCK128 [E_local, K/128, N] or PER_TENSOR [1]).  Groups,
 * group_offset and E_local are as in gmm_fp8: rows outside the local groups
 * are zero.
 *
 * The contraction runs on the f16 tensor-core MMA (both code types are exact
 * in f16) with fp32 accumulation.  Blockwise weight scales enter as factors
 * s_w[kb] / max_kb s_w[kb] on the converted codes, so each converted weight
 * carries one f16 rounding (relative 2^-12; coarser where the factor falls
 * below 2^-14, the f16 normal range) beside the fp32 accumulation.
 *
 * workspace (optional, may be NULL): caller-owned device memory of at least
 * gmm_fp8_w8_workspace_bytes(M, K) bytes, 16-byte aligned.  Where the local
 * groups average 256 rows or more (the tensor pipe binds), the call then
 * first decodes lhs_q to f16 there (one pass over the codes) and the
 * contraction reads the f16 rows directly; otherwise, and without a
 * workspace, the contraction converts the e4m3 codes on the SM.  The result
 * is the same, bit for bit.
 * K % 16 == 0 (% 128 for blockwise), N % 16 == 0; lhs_q, rhs_q and out
 * 16-byte aligned.  MOE_ERR_INVALID_ARG on a bad argument (a workspace too
 * small or misaligned included), before any launch. */
moe_status gmm_fp8_w8(const uint8_t* lhs_q, const float* lhs_scale, moe_scale_mode lhs_mode, const int8_t* rhs_q,
                      const float* rhs_scale, moe_scale_mode rhs_mode, const int32_t* group_sizes, int E,
                      int group_offset, int E_local, int64_t M, int64_t K, int64_t N, uint16_t* out,
                      void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Bytes of gmm_fp8_w8's optional workspace: 2 * M * K (0 for an empty or
 * out-of-range shape). */
size_t gmm_fp8_w8_workspace_bytes(int64_t M, int64_t K);

#ifdef __cplusplus
}
#endif

#endif /* MOEFP8_H_ */
