/*
 * moe.h -- C ABI of libmoe_gb300.so: the single-GPU forward of one
 * Mixture-of-Experts FFN layer on GB300 (sm_103a).
 *
 * The layer, as the page "MOE推理流程解析" (ffner.com) lays it out:
 *   section 三: the router scores every eligible expert; top-k keeps the
 *     chosen experts' indices and weights; a permutation reads the token
 *     vectors, writes them in expert order and records an inverse map; a
 *     grouped GEMM runs all expert matrices (of different row counts) in
 *     one launch; each expert applies its activation and output projection;
 *     the inverse map restores token order, the routing weight is applied
 *     and the contributions of the same token are summed.
 *   section 二: assignments (token vector, expert, weight) are grouped by
 *     expert into contiguous matrices, each row keeping its source token id;
 *     an expert batch counts assignments, not unique tokens (top-2 gives two
 *     rows per token).
 *   section 一: shared experts process every token whatever the router
 *     scores.
 * Precision ("MoE 推理部署", zzmblog.top, section 专家量化): quantisation
 * scales are per expert; the router and shared experts stay at higher
 * precision than quantised routed experts.
 *
 * Conventions (all entry points)
 *   - Every pointer named as a tensor is a DEVICE pointer of the current CUDA
 *     device, row-major, densely packed, 16-byte aligned.  The caller owns
 *     every buffer and the stream; the library allocates no device memory.
 *   - Weights are [out, in] (the reduction index is contiguous):
 *       w_router [E, d]; w_gate, w_up [E, ffn, d]; w_down [E, d, ffn];
 *       shared expert: w_shared_gate, w_shared_up [ffn_shared, d],
 *       w_shared_down [d, ffn_shared].
 *   - Experts are numbered from 0.  R = T * k assignment rows.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     Argument errors are detected on the host and returned before anything
 *     is enqueued; launch failures return MOE_ERR_CUDA.  Errors found by a
 *     kernel (an expired bounded wait, an out-of-range index) are recorded in
 *     a per-device status word read by moe_read_device_status().
 *   - Unsupported combinations of sizes or dtypes return MOE_ERR_UNSUPPORTED;
 *     there is no fallback path.
 *   - T == 0 is valid: nothing is enqueued and MOE_OK is returned.
 *
 * Supported storage:  act_dtype / w_dtype
 *   MOE_F32  / MOE_F32          fp32 CUDA-core path (fp32 accumulation)
 *   MOE_BF16 / MOE_BF16         tcgen05 tensor-core path (fp32 accumulation)
 *   MOE_BF16 / MOE_FP8_E4M3     as above, FP8 weights (OCP E4M3) with fp32
 *                               per-expert, per-output-channel scales;
 *                               the router and shared expert stay bf16.
 *                               The bf16 rows (tokens, then h) enter the
 *                               FP8 x FP8 tensor-core instructions as two
 *                               E4M3 rows each (moe_split_rows_e4m3x2),
 *                               the bf16 values themselves for elements
 *                               within 2^9 of their row's maximum:
 *                               g[r,o] = s_gate[e,o] * s_x[r] *
 *                                 sum_i (hi[r,i] + lo[r,i]) code_gate[e][o,i]
 *                               (likewise u); h = SiLU(g) * u held in bf16,
 *                               split the same way before the down product.
 *                               Any finite bf16 magnitude is accepted.
 *   MOE_BF16 / MOE_FP8_E4M3_ACT8
 *                               FP8 weights as above; both routed GEMMs
 *                               multiply them with E4M3 activation rows
 *                               (per-row scales, moe_quantize_rows_e4m3):
 *                               g[r,o] = s_x[r] * s_gate[e,o] *
 *                                        sum_i q_x[r,i] * code_gate[e][o,i]
 *                               (likewise u), h = SiLU(g) * u held in f16
 *                               and quantised per row the same way, then
 *                               y[r,o] = s_h[r] * s_down[e,o] *
 *                                        sum_j q_h[r,j] * code_down[e][o,j].
 *                               Router and shared expert stay bf16.
 *   MOE_BF16 / MOE_MXFP4        OCP Microscaling FP4 weights ("MoE 推理部署",
 *                               section 专家量化: MXFP4 block-scaled 4-bit
 *                               experts): W[o,i] = E2M1(code[o,i]) *
 *                               2^(s[i/32,o] - 127).  w_gate / w_up
 *                               [E, ffn, d/2] and w_down [E, d, ffn/2] bytes,
 *                               two codes per byte (element 2i in the low
 *                               nibble of byte i); s_gate / s_up [E, d/32,
 *                               ffn] and s_down [E, ffn/32, d] UE8M0 bytes,
 *                               reduction-block-major (a k-block's scales of
 *                               all output channels contiguous), passed
 *                               through the float* scale parameters.  The
 *                               kernels convert to f16 operands, exactly for
 *                               block scales 2^-23 .. 2^13 (UE8M0 104..140);
 *                               larger scales overflow f16 and are not
 *                               supported.  Router and shared expert bf16.
 * Size limits: 1 <= k <= min(E, 32), E <= 1024, T * k <= 2^24,
 * d % 8 == 0, ffn % 8 == 0; the tensor-core path further needs
 * d % 128 == 0, ffn % 128 == 0 and ffn_shared % 128 == 0.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 5

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* A cudaStream_t. */
typedef struct CUstream_st *moe_stream_t;

typedef enum moe_dtype {
  MOE_F32 = 0,
  MOE_BF16 = 1,
  MOE_FP8_E4M3 = 2,
  /* w_dtype only: FP8 weights as MOE_FP8_E4M3, and both routed expert
   * products take activations quantised per row to E4M3
   * (moe_quantize_rows_e4m3) on FP8 x FP8 tensor-core instructions */
  MOE_FP8_E4M3_ACT8 = 3,
  /* w_dtype only: OCP MXFP4 routed expert weights (see "Supported storage") */
  MOE_MXFP4 = 4
} moe_dtype;

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,    /* null pointer, bad size, k > E, ...        */
  MOE_ERR_UNSUPPORTED = -2,    /* valid but not implemented combination     */
  MOE_ERR_WORKSPACE = -3,      /* workspace missing or too small            */
  MOE_ERR_CUDA = -4,           /* a CUDA runtime / driver call failed       */
  MOE_ERR_DEVICE_TIMEOUT = -5, /* a kernel's bounded wait expired           */
  MOE_ERR_DEVICE_BOUNDS = -6   /* a kernel met an out-of-range index/offset */
} moe_status;

/* The problem statement shared by every entry point. */
typedef struct moe_problem {
  int32_t T;          /* tokens in the batch                                */
  int32_t d;          /* hidden size                                        */
  int32_t ffn;        /* routed expert intermediate size                    */
  int32_t E;          /* routed experts                                     */
  int32_t k;          /* experts chosen per token                           */
  int32_t ffn_shared; /* shared expert intermediate size; 0 = none          */
  int32_t act_dtype;  /* moe_dtype of x, w_router, shared expert, outputs   */
  int32_t w_dtype;    /* moe_dtype of the routed expert weights             */
} moe_problem;

/*
 * moe_router_topk -- router scores, softmax, top-k, renormalised weights.
 * Page "MOE推理流程解析", section 三 (the router scores each eligible expert;
 * top-k keeps the chosen indices and weights) and section 九 (the kept
 * weights are re-normalised).
 *
 *   l[t,e]   = sum_i x[t,i] * w_router[e,i] (+ router_bias[e]), fp32 accumulate
 *   p        = softmax(l[t,:]) over all E experts
 *   S_t      = the k experts with the largest l (ties: lower expert index)
 *   w[t,j]   = p[S_t,j] / sum_{e in S_t} p[e]   (== softmax over S_t only)
 * Slots j are in descending weight.  Non-finite logits: infinities order as
 * numbers, -0 ties +0, and NaN logits rank after every number (among
 * themselves by expert index).
 *
 *   x            [T, d] act_dtype
 *   w_router     [E, d] act_dtype
 *   router_bias  [E] fp32 or NULL
 *   logits_in    [T, E] fp32 or NULL: when given, used as l directly (no
 *                matmul; router_bias must then be NULL; x, w_router unused)
 *   logits_out   [T, E] fp32 or NULL: receives l (including the bias)
 *   topk_idx     [T, k] int32 out      topk_w  [T, k] fp32 out
 */
MOE_API moe_status moe_router_topk(const moe_problem *p, const void *x, const void *w_router,
                           const float *router_bias, const float *logits_in,
                           float *logits_out, int32_t *topk_idx, float *topk_w,
                           moe_stream_t stream);

/*
 * moe_permute -- group the T*k assignments by expert and move token rows.
 * Page "MOE推理流程解析", section 二 (grouping by expert into contiguous
 * matrices, the source token id kept beside each row) and section 三 (the
 * permutation writes token vectors in expert order and records an inverse
 * map for the combine).
 *
 *   counts[e]       = #{(t,j) : topk_idx[t,j] == e}                [E] int32 out
 *   offsets[e]      = sum_{e'<e} counts[e'], offsets[E] = T*k     [E+1] int32 out
 *   perm_token[r]   = source token of row r                       [T*k] int32 out
 *   inv_row[t*k+j]  = row holding assignment (t, j)               [T*k] int32 out
 *   x_perm[r, :]    = x[perm_token[r], :]      [T*k, d] act_dtype out, or NULL
 * Rows inside an expert's range are in ascending token order (deterministic,
 * bit-exact).  x may be NULL only when x_perm is NULL.  topk_idx entries
 * outside [0, E) are skipped and flag MOE_ERR_DEVICE_BOUNDS.
 * workspace: at least moe_workspace_size() bytes, device memory.
 */
MOE_API moe_status moe_permute(const moe_problem *p, const int32_t *topk_idx, const void *x,
                       int32_t *counts, int32_t *offsets, int32_t *perm_token,
                       int32_t *inv_row, void *x_perm, void *workspace,
                       size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_permute_static_scratch -- moe_permute without a workspace argument.
 * No counterpart on the pages: it exists for callers that cannot allocate
 * device memory -- code hosted by another framework whose memory manager
 * must own every allocation, or latency-critical loops that cannot afford a
 * cudaMalloc (which may synchronise the device).  Arguments and results are
 * those of moe_permute; the caller still passes every input and output.
 *
 * The scratch moe_permute takes from the workspace (per-chunk expert counts,
 * ceil(T*k/256) * E int32 values) lives instead in a 1 MiB array compiled
 * into the library and held by every GPU that loads it until the process
 * exits.  Problems needing more (ceil(T*k/256) * E > 262144) are rejected
 * with MOE_ERR_WORKSPACE.  The first call on each device looks up the
 * array's device address with that device current; make that first call
 * before any stream capture.  That cached address (like the library's other
 * per-device state) does not survive a device reset (cudaDeviceReset) in
 * the same process.  The problem is checked exactly as moe_permute checks
 * it, then against the array's size.  All calls share the array and it keeps the
 * last call's contents (every entry read is first rewritten, so nothing has
 * to be cleared); calls that overlap on the GPU race on it.  Allocates
 * nothing.
 */
MOE_API moe_status moe_permute_static_scratch(const moe_problem *p, const int32_t *topk_idx,
                                              const void *x, int32_t *counts, int32_t *offsets,
                                              int32_t *perm_token, int32_t *inv_row,
                                              void *x_perm, moe_stream_t stream);

/*
 * moe_grouped_swiglu -- all expert matrices in one grouped computation.
 * Page "MOE推理流程解析", section 三 (a grouped GEMM runs several expert
 * matrices with different row counts in one launch; each expert applies its
 * activation and output projection) and section 二 (variable-row expert
 * matrices, no padding in the result).
 *
 * For every expert e and every row r in [offsets[e], offsets[e+1]):
 *   h[r,:]      = SiLU(x_perm[r,:] W_g[e]^T) * (x_perm[r,:] W_u[e]^T)
 *   y_perm[r,:] = h[r,:] W_d[e]^T
 * with FP8 weights W[e][o,:] = code[e][o,:] * scale[e][o] (s_gate, s_up
 * [E, ffn]; s_down [E, d]; NULL unless the weights are quantised: FP8, or
 * MXFP4 with the block-scale arrays described above).  With
 * MOE_FP8_E4M3_ACT8 the rows of x_perm and of h enter their products
 * quantised per row (moe_quantize_rows_e4m3, into the workspace).
 *
 *   x_perm   [T*k, d] act_dtype      offsets [E+1] int32 (device)
 *   y_perm   [T*k, d] act_dtype out
 * h is kept in workspace in act_dtype (bf16 for the tensor-core path).
 * Offsets must be non-decreasing with offsets[E] <= T*k; rows outside every
 * expert's range are left untouched.
 */
MOE_API moe_status moe_grouped_swiglu(const moe_problem *p, const void *x_perm, const int32_t *offsets,
                              const void *w_gate, const void *w_up, const void *w_down,
                              const float *s_gate, const float *s_up, const float *s_down,
                              void *y_perm, void *workspace, size_t workspace_bytes,
                              moe_stream_t stream);

/*
 * moe_quantize_rows_e4m3 -- per-row FP8 quantisation of activation rows.
 * Page "MOE推理流程解析", section 三 (activations may be quantised before
 * dispatch, so that the permuted rows move fewer bytes, or dispatched at
 * higher precision and quantised just before the experts) and page
 * "MoE 推理部署", section 专家量化 (FP8 inference).  The layer forward with
 * w_dtype MOE_FP8_E4M3_ACT8 quantises x before dispatch with this
 * operation, moe_grouped_swiglu quantises x_perm (after dispatch), and both
 * quantise the rows of h (held in f16) before the down product.
 *
 *   s[r]      = max_i |x[r,i]| / 448, or 1 when row r is all zero
 *   code[r,i] = E4M3(x[r,i] / s[r]): nearest E4M3 value, ties to the even
 *               code, magnitudes above 448 saturated to 448, sign kept
 *               (-0 -> 0x80)
 * Both divisions are correctly rounded fp32 operations, so the codes and
 * scales are exact functions of the inputs (bit-reproducible).
 *
 *   x       [rows, cols] bf16, device, 16-byte aligned
 *   codes   [rows, cols] uint8 out (OCP E4M3 bit patterns), 16-byte aligned
 *   scales  [rows] fp32 out
 * rows >= 0 (0: nothing is enqueued); cols > 0 and cols % 8 == 0, else
 * MOE_ERR_UNSUPPORTED.  Null pointers with rows > 0: MOE_ERR_INVALID_ARG.
 */
MOE_API moe_status moe_quantize_rows_e4m3(int32_t rows, int32_t cols, const void *x, uint8_t *codes,
                                          float *scales, moe_stream_t stream);

/*
 * moe_split_rows_e4m3x2 -- bf16 rows as two E4M3 rows each, exactly.
 * Page "MoE 推理部署", section 专家量化 (FP8 expert weights, the
 * activations kept at higher precision): the FP8-weight mode
 * (MOE_FP8_E4M3) multiplies its E4M3 weights with bf16 activation rows on
 * FP8 x FP8 tensor-core instructions by handing them each row in this
 * form; the layer forward applies it to x (before dispatch) and to h.
 *
 *   s[r]         = 2^p, p the integer with max_i |x[r,i]| / 2^p in
 *                  (224, 448]; 1 when row r is all zero
 *   hi[r,i]      = E4M3(x[r,i] / s[r])
 *   lo[r,i]      = E4M3(x[r,i] / s[r] - hi[r,i])
 * (nearest E4M3 value, ties to the even code).  Then
 *   x[r,i] = s[r] * (hi[r,i] + lo[r,i])
 * exactly for every element with |x[r,i]| >= max_i |x[r,i]| * 2^-9, and
 * within s[r] * 2^-10 for smaller ones: a bf16 value has 8 significant
 * bits, hi holds the top four (rounded) and lo the signed remainder, which
 * E4M3 holds exactly down to its smallest step.  An FP8 x FP8 product on
 * hi plus one on lo, accumulated together, multiplies by the bf16 row.
 *
 *   x       [rows, cols] bf16, device, 16-byte aligned
 *   codes   [2, rows, cols] uint8 out: every row's hi codes, then every
 *           row's lo codes (row r's lo codes are row rows + r of a
 *           [2*rows, cols] matrix), 16-byte aligned
 *   scales  [rows] fp32 out (powers of two)
 * rows >= 0 (0: nothing is enqueued); cols > 0 and cols % 8 == 0, else
 * MOE_ERR_UNSUPPORTED.  Null pointers with rows > 0: MOE_ERR_INVALID_ARG.
 */
MOE_API moe_status moe_split_rows_e4m3x2(int32_t rows, int32_t cols, const void *x, uint8_t *codes,
                                         float *scales, moe_stream_t stream);

/*
 * moe_combine -- restore token order, apply routing weights, sum.
 * Page "MOE推理流程解析", section 三 (the inverse map restores token order,
 * the routing weight is applied, contributions with the same token id are
 * summed) and section 二 (T1's output is 0.7 * E1(T1) + 0.3 * E3(T1)).
 *
 *   out[t,:] = sum_{j<k} topk_w[t,j] * y_perm[inv_row[t*k+j], :] (+ shared_out[t,:])
 * accumulated in fp32 in slot order j = 0..k-1, rounded once to act_dtype.
 *   y_perm [T*k, d]  inv_row [T*k] int32  topk_w [T, k] fp32
 *   shared_out [T, d] act_dtype or NULL      out [T, d] act_dtype
 */
MOE_API moe_status moe_combine(const moe_problem *p, const void *y_perm, const int32_t *inv_row,
                       const float *topk_w, const void *shared_out, void *out,
                       moe_stream_t stream);

/*
 * moe_layer_forward -- the whole layer: router top-k, permutation, grouped
 * SwiGLU experts, optional shared expert, combine (page "MOE推理流程解析",
 * sections 一, 二, 三; section 十一 lists the step: routing, token
 * permutation, grouped expert compute, combine, unpermutation).
 *
 *   out[t,:] = sum_{e in S_t} w[t,e] * FFN_e(x[t,:]) + FFN_shared(x[t,:])
 *
 * Shared expert weights are all NULL when p->ffn_shared == 0, all non-NULL
 * otherwise.  topk_idx_out [T,k], topk_w_out [T,k] and counts_out [E] are
 * optional copies of the routing decision (NULL = not wanted).
 * The whole sequence is enqueued on `stream` without any host
 * synchronisation, so it can be captured into a CUDA graph by the caller.
 */
MOE_API moe_status moe_layer_forward(const moe_problem *p, const void *x, const void *w_router,
                             const float *router_bias, const void *w_gate, const void *w_up,
                             const void *w_down, const float *s_gate, const float *s_up,
                             const float *s_down, const void *w_shared_gate,
                             const void *w_shared_up, const void *w_shared_down, void *out,
                             int32_t *topk_idx_out, float *topk_w_out, int32_t *counts_out,
                             void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * Per-stage timing of the layer forward (page "MOE推理流程解析", section 三:
 * measure routing, permutation, expert GEMM and combine separately; one
 * merged MoE timer cannot say which stage is slow).
 *
 * A stage timer holds CUDA events for one call of moe_layer_forward_timed();
 * reading it waits for that call's last event.  Stage indices:
 */
enum {
  MOE_STAGE_ROUTER = 0,   /* logits, softmax, top-k                        */
  MOE_STAGE_PERMUTE = 1,  /* counts, offsets, maps, row moves              */
  MOE_STAGE_GATE_UP = 2,  /* grouped gate/up GEMM + SiLU*mul               */
  MOE_STAGE_DOWN = 3,     /* grouped down GEMM                             */
  MOE_STAGE_SHARED = 4,   /* shared expert (0 when absent)                 */
  MOE_STAGE_COMBINE = 5,  /* unpermute, weights, sum                       */
  MOE_NUM_STAGES = 6
};
typedef struct moe_stage_timer moe_stage_timer;

/* Create / destroy a timer (host object owning CUDA events; no device memory). */
MOE_API moe_status moe_stage_timer_create(moe_stage_timer **timer);
MOE_API moe_status moe_stage_timer_destroy(moe_stage_timer *timer);
/* Wait for the timed call to finish; ms[MOE_NUM_STAGES] receives each stage's
 * device time in milliseconds. */
MOE_API moe_status moe_stage_timer_read(moe_stage_timer *timer, float *ms);

/* moe_layer_forward with CUDA events recorded on `stream` between stages. */
MOE_API moe_status moe_layer_forward_timed(
    const moe_problem *p, const void *x, const void *w_router, const float *router_bias,
    const void *w_gate, const void *w_up, const void *w_down, const float *s_gate,
    const float *s_up, const float *s_down, const void *w_shared_gate, const void *w_shared_up,
    const void *w_shared_down, void *out, int32_t *topk_idx_out, float *topk_w_out,
    int32_t *counts_out, void *workspace, size_t workspace_bytes, moe_stream_t stream,
    moe_stage_timer *timer);

/* Number of kernels one moe_layer_forward() call launches for problem *p on
 * the current device (written to *launches). */
MOE_API moe_status moe_layer_launch_count(const moe_problem *p, int32_t *launches);

/*
 * moe_plan_info -- the tiling the library chose for problem *p on the
 * current device (no page counterpart; for benchmarks and tests):
 * info[0] rows per tile of the gate/up GEMM, info[1] rows per tile of the
 * down GEMM, info[2] reduction splits of the down GEMM, info[3] persistent
 * CTAs per GEMM launch, info[4] reduction splits of the gate/up GEMM,
 * info[5] bit 0 / bit 1: the gate/up / down GEMM runs on CTA pairs
 * (256 output channels per tile).  `info` holds 6 entries.  All zero for
 * the fp32 CUDA-core path.
 */
MOE_API moe_status moe_plan_info(const moe_problem *p, int32_t *info);

/*
 * moe_plan_info_for, moe_layer_launch_count_for, moe_workspace_size_for --
 * the same answers as moe_plan_info, moe_layer_launch_count and
 * moe_workspace_size for a device with `num_sms` multiprocessors, computed
 * on the host alone: they touch no device and need none (planning ahead of
 * time, and tests of the tiling rules on machines without a GPU).  The
 * device entry points are these with the current device's SM count.
 * Returns MOE_ERR_INVALID_ARG for a null output or num_sms outside
 * [1, 4096], and MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for problems the
 * library rejects.
 */
MOE_API moe_status moe_plan_info_for(const moe_problem *p, int32_t num_sms, int32_t *info);
MOE_API moe_status moe_layer_launch_count_for(const moe_problem *p, int32_t num_sms, int32_t *launches);
MOE_API moe_status moe_workspace_size_for(const moe_problem *p, int32_t num_sms, size_t *bytes);

/*
 * moe_workspace_size -- device workspace (bytes) sufficient for every entry
 * point above with problem *p on the current device.  Returns
 * MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for problems the library rejects.
 */
MOE_API moe_status moe_workspace_size(const moe_problem *p, size_t *bytes);

/*
 * moe_read_device_status -- synchronise `stream`, then read and clear the
 * current device's kernel status word.  *status receives MOE_OK or the first
 * error a kernel recorded since the last read (MOE_ERR_DEVICE_TIMEOUT,
 * MOE_ERR_DEVICE_BOUNDS).  Returns MOE_ERR_CUDA if synchronisation fails.
 */
MOE_API moe_status moe_read_device_status(moe_stream_t stream, int32_t *status);

/* Human-readable name of a status code (static storage). */
MOE_API const char *moe_status_string(int32_t status);

/* The last CUDA error text recorded by a call that returned MOE_ERR_CUDA on
 * this host thread (static thread-local storage; "" if none). */
MOE_API const char *moe_last_cuda_error(void);

/* MOE_ABI_VERSION of the loaded library. */
MOE_API int32_t moe_abi_version(void);

/*
 * moe_selftest_bounded_wait -- failure-detection self test (no page
 * counterpart).  Launches the tensor-core kernel's wait machinery on a
 * barrier that nothing arrives at, with a wait limit of timeout_ns
 * nanoseconds.  No copy or MMA is issued, so the wait expiring leaves no
 * work in flight; the kernel records MOE_ERR_DEVICE_TIMEOUT in the status
 * word, frees its tensor memory and returns.  Read the outcome with
 * moe_read_device_status().
 */
MOE_API moe_status moe_selftest_bounded_wait(int64_t timeout_ns, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
