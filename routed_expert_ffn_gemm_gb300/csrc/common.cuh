// Internal declarations shared by the translation units of libmoe_gb300.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// host-side context
// ---------------------------------------------------------------------------

struct DeviceCtx {
  int device = -1;
  int num_sms = 0;
  int* status = nullptr;  // device address of this device's status word
  // side stream + fork/join events (created on first use): the layer runs
  // the shared expert there, concurrently with routing and permutation
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

// Current device, its SM count and status-word address (cached per device).
// The cache outlives a device reset (cudaDeviceReset) in the same process,
// so the library is not usable after one.
moe_status device_ctx(DeviceCtx* ctx);

// The checks every entry point that takes a moe_problem applies (sizes,
// dtype combination, divisibility, router limits): MOE_OK, or the status
// the entry point returns before launching anything.
moe_status problem_check(const moe_problem* p);

// Remember the text of a failed CUDA call for moe_last_cuda_error().
void record_cuda_error(cudaError_t err);
void record_cuda_error_text(const char* text);

inline moe_status cuda_status(cudaError_t err) {
  if (err == cudaSuccess) return MOE_OK;
  record_cuda_error(err);
  return MOE_ERR_CUDA;
}

#define MOE_TRY_CUDA(expr)                                   \
  do {                                                       \
    cudaError_t _e = (expr);                                 \
    if (_e != cudaSuccess) return ::moe::cuda_status(_e);    \
  } while (0)

#define MOE_TRY(expr)                                        \
  do {                                                       \
    moe_status _s = (expr);                                  \
    if (_s != MOE_OK) return _s;                             \
  } while (0)

// 2-D row-major tensor map for TMA: `rows` x `cols` elements of
// `elem_bytes` (2: bf16, 1: bytes), row pitch `cols * elem_bytes`, box
// `box_cols` x `box_rows`, swizzle of `swizzle_bytes` (128, 64 or 0: none),
// zero fill out of bounds.
moe_status make_tmap_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                        int elem_bytes, uint32_t box_rows, uint32_t box_cols, int swizzle_bytes);
// 3-D view of the same row-major matrix (16-bit elements, cols % 128 == 0)
// whose box {64, box_rows, 2} copies two consecutive 64-element column
// blocks at once, as two 128-byte-swizzled tiles one after the other.
moe_status make_tmap_kpair(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           int elem_bytes, uint32_t box_rows);

// ---------------------------------------------------------------------------
// launches: programmatic dependent launch
// ---------------------------------------------------------------------------

// Every kernel of the library is launched with programmatic stream
// serialisation: it may be scheduled while the previous kernel on the stream
// is still finishing, and it calls griddep_wait() before its first access to
// global memory, which returns once the previous grid has completed and its
// writes are visible.  This overlaps launch latency and kernel prologues with
// the previous kernel's tail.  MOE_PDL=0 in the environment launches plainly.
bool pdl_enabled();

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kc(int cluster, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {  // thread-block clusters of `cluster` CTAs along x
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args&&... args) {
  return launch_kc(1, kern, grid, block, smem, s, std::forward<Args>(args)...);
}

// Record `ev` on `s`; inside stream capture as an external (timestamp) node,
// so a captured layer keeps its stage times.
inline cudaError_t record_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &st);
  if (e != cudaSuccess) return e;
  return st == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                             : cudaEventRecord(ev, s);
}

// Wait until the previous grid on the stream has completed (no-op when the
// kernel was not launched as a programmatic dependent).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next grid on the stream be scheduled (it still waits in
// griddep_wait() for this grid to complete).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_begin() {
  griddep_wait();
  griddep_launch_dependents();
}

// ---------------------------------------------------------------------------
// device-side status word
// ---------------------------------------------------------------------------

// Record the first error of a kernel (the status word keeps the first one).
__device__ __forceinline__ void set_device_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// kernel launchers (each in its own translation unit)
// ---------------------------------------------------------------------------

struct RouterArgs {
  int T, d, E, k, act_dtype;
  const void* x;
  const void* w_router;
  const float* bias;
  const float* logits_in;
  float* logits_out;
  int32_t* idx;
  float* w;
  // tensor-core logits (bf16, E % 128 == 0, large T): scratch of
  // tc_splits * T * E fp32 (may be logits_out when tc_splits == 1)
  float* tc_scratch;
  int tc_splits;
  int num_sms;
  int* status;
  // 1: when the top-k would be a separate pass over global logits, skip it
  // (the caller's permutation selects the top-k from logits_out itself)
  int defer_topk;
};
// Tensor-core logits apply to this problem (and how many K splits), given a
// scratch of `scratch_floats` fp32 values; 0 = use the CUDA-core kernels.
int router_tc_splits(int T, int d, int E, int act_dtype, int num_sms, size_t scratch_floats);
moe_status router_topk_launch(const RouterArgs& a, cudaStream_t s);
moe_status router_topk_check(int d, int E, int act_dtype);
int router_launch_count(int T, int E, bool logits_in, bool logits_out);
// The CUDA-core router writes global logits and selects the top-k in a
// separate pass (the pass `defer_topk` skips).
bool router_topk_separate(int T, int E, bool logits_in, bool logits_out);

struct PermuteArgs {
  int T, k, E, d, act_bytes;
  const int32_t* idx;
  const void* x;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm_token;
  int32_t* inv_row;
  void* x_perm;
  int32_t* chunk_scratch;  // [n_chunks * E] when the chunked path is used
  int* status;
  int to_f16;              // 1: x is bf16 and x_perm receives it rounded to f16
  // nullable: router logits [T, E]; the small path then selects the top-k
  // itself into idx_out / w_out (and reads idx from there)
  const float* topk_logits;
  int32_t* idx_out;
  float* w_out;
  // nullable: zero_n int32 the first permutation kernel sets to zero
  int32_t* zero;
  size_t zero_n;
};
// Largest T*k the single-block path (which can also select the top-k) takes.
int permute_small_max();
size_t permute_scratch_bytes(int T, int k, int E);
int permute_launch_count(int T, int k, bool move_rows);
moe_status permute_launch(const PermuteArgs& a, cudaStream_t s);
// bf16 rows -> f16 rows (saturating), n elements, n % 8 == 0.
moe_status bf16_to_f16_launch(const void* src, void* dst, size_t n, cudaStream_t s);
// Per-row E4M3 codes [rows, d] and fp32 scales [rows] of 16-bit rows x
// (bf16, or f16 with f16_in; scale = row absmax / 448): the FP8-activation
// mode's operands of both expert GEMMs.
moe_status quantize_rows_e4m3_launch(const void* x, int rows, int d, void* codes, float* scales,
                                     int num_sms, cudaStream_t s, bool f16_in = false);
// Two-term E4M3 encoding of 16-bit rows (bf16, or f16 with f16_in): codes
// [2, rows, d] (every row's hi codes, then every row's lo codes) and
// power-of-two scales [rows] with x = s * (hi + lo), exact for elements
// within 2^9 of the row's largest magnitude: the operands of FP8-weight
// GEMMs on bf16 activations.
moe_status split_rows_e4m3x2_launch(const void* x, int rows, int d, void* codes, float* scales, int num_sms,
                                    cudaStream_t s, bool f16_in = false);
// The same split of bf16 token rows x [T, d], each written to its k rows of
// the permuted order (dst_rows [T*k]: inv_row) of codes [2, R, d] and
// scales [R]: the B operand of a gate/up GEMM that loads rows by TMA tiles
// instead of gathering them.
moe_status split_rows_e4m3x2_scatter_launch(const void* x, int T, int d, int k, const int32_t* dst_rows, int R,
                                            void* codes, float* scales, int* status, int num_sms,
                                            cudaStream_t s);

struct CombineArgs {
  int T, k, d, act_dtype;
  const void* y;           // y_perm [R, d] act dtype, or fp32 partials
  int y_partials;          // 0: y is act dtype [R, d]; S>0: fp32 [S, R, d]
  const int32_t* inv_row;
  const float* w;
  const void* shared;      // [T, d] act dtype or nullptr
  void* out;
};
moe_status combine_launch(const CombineArgs& a, cudaStream_t s);

// fp32 CUDA-core grouped SwiGLU (both GEMMs, fp32 accumulation).
struct SimtGroupedArgs {
  int R, d, ffn, E;
  const float* x_perm;
  const int32_t* offsets;
  const float* w_gate;
  const float* w_up;
  const float* w_down;
  float* h;       // [R, ffn] scratch
  float* y;       // [R, d]
  int* status;
};
// `mid` (nullable): event recorded between the gate/up and the down kernels.
moe_status simt_grouped_launch(const SimtGroupedArgs& a, cudaStream_t s, cudaEvent_t mid);

// tcgen05 grouped GEMM (bf16 or FP8 weights, bf16 activations).
struct TcPlan {
  int bn_gateup;       // max rows per tile in the gate/up GEMM
  int bn_down;         // max rows per tile in the down GEMM
  int splits_down;     // K splits of the down GEMM (1 = direct bf16 output)
  int splits_gateup;   // K splits of the gate/up GEMM (1 = SiLU*mul in its epilogue;
                       // else fp32 partials, then an in-order sum + SiLU*mul pass)
  int grid;            // persistent CTAs
  int pair_gateup;     // 1: the gate/up GEMM runs on CTA pairs (cta_group::2, M = 256)
  int pair_down;       // 1: the down GEMM runs on CTA pairs
  int boxn_gateup;     // rows per TMA box of the B rows (tile loads), gate/up and down
  int boxn_down;
};
struct TcGroupedArgs {
  int R, d, ffn, G;    // rows, hidden, intermediate, groups (experts)
  int w_dtype;         // MOE_BF16, MOE_FP8_E4M3 or MOE_FP8_E4M3_ACT8
  const void* x_perm;  // [R, d] B operand of gate/up: bf16, or f16 with FP8 weights
  const int32_t* offsets;
  const void* w_gate;
  const void* w_up;
  const void* w_down;
  const float* s_gate;
  const float* s_up;
  const float* s_down;
  void* h;             // [R, ffn] scratch: bf16, or f16 with FP8 weights
  void* y;             // [R, d] bf16 when splits_down == 1, else fp32 [S, R, d]
  int* status;
  long long timeout_ns;
  // nullable: gather the gate/up row operand from x_src [T_src, d] (rows
  // gather_rows[r], e.g. perm_token) instead of reading x_perm
  const int32_t* gather_rows;
  const void* x_src;
  int T_src;
  float* gu_partials;  // [splits_gateup, R, 2*ffn] fp32 when splits_gateup > 1
  // nullable with gu_partials: zeroed arrival counters (gu_counters_size
  // ints); the GEMM then finalizes h itself instead of a separate pass
  int* gu_cnt;
  // FP8 activations (w_dtype MOE_FP8_E4M3_ACT8): x_perm / x_src hold E4M3
  // codes and row_scale their per-row scales ([T_src] with gather_rows,
  // else [R]); h_q [R, ffn] / h_scale [R] receive h's codes and row scales
  // for the down GEMM
  const float* row_scale;
  void* h_q;
  float* h_scale;
  // 1: the offsets and the weights are complete before gate/up's grid
  // passes its griddepcontrol.wait (the layer: the permutation wrote the
  // offsets), so the down GEMM requests its first weight tiles before its
  // own wait (TcParams::early_w)
  int early_down;
};
// FP8 weights with bf16 activations run on two-term E4M3 rows (the default;
// MOE_FP8_CONVERT=1 selects the E4M3 -> f16 weight converters instead).
bool fp8_two_term(int w_dtype);
// Whether the layer hands the gate/up GEMM of this plan two-term rows in
// permuted order (tile loads) rather than per token (gathered rows): at
// prefill tiles, where gathering two rows per row costs the producer more
// than the one scatter pass.
bool fp8_two_term_scattered(int w_dtype, const TcPlan& plan);
// Arrival counters the fused gate/up finalize needs for R rows in G groups.
size_t gu_counters_size(int R, int G, int ffn, const TcPlan& plan);
TcPlan tc_plan(int T, int k, int E, int d, int ffn, int num_sms, int w_dtype);
moe_status tc_grouped_launch(const TcGroupedArgs& a, const TcPlan& plan, cudaStream_t s,
                             cudaEvent_t mid);
moe_status tc_selftest_launch(int* status, long long timeout_ns, cudaStream_t s);
// Dense out[s][n][m] = sum over the s-th K slice of a[m, :] . b[n, :] (bf16
// operands, fp32 results, `splits` K slices), on the tensor cores.
moe_status tc_dense_f32_launch(const void* a, const void* b, float* out, int M, int N, int K,
                               int splits, int num_sms, int* status, long long timeout_ns,
                               cudaStream_t s);

// Default limit of every bounded wait inside a kernel (nanoseconds).
constexpr long long kDefaultWaitNs = 2000000000LL;

}  // namespace moe
