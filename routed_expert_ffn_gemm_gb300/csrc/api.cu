// C-ABI entry points: host-side validation, workspace layout, and the
// launch sequence of the layer forward ("MOE推理流程解析", section 三 and
// section 十一: routing, token permutation, grouped expert compute, combine,
// unpermutation; every stage on one GPU, section 二).
#include <stdlib.h>

#include "common.cuh"

namespace moe {
namespace {

size_t act_bytes(int dt) { return dt == MOE_F32 ? 4 : 2; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Which compute path a problem takes.
enum class Path { kSimt, kTensor };

moe_status check_problem(const moe_problem* p, Path* path) {
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  if (p->T < 0 || p->d <= 0 || p->ffn <= 0 || p->E <= 0 || p->k <= 0 || p->ffn_shared < 0)
    return MOE_ERR_INVALID_ARG;
  if (p->k > p->E) return MOE_ERR_INVALID_ARG;
  if (p->k > 32 || p->E > 1024) return MOE_ERR_UNSUPPORTED;
  if (p->d % 8 != 0 || p->ffn % 8 != 0 || p->ffn_shared % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)p->T * p->k > (1 << 24)) return MOE_ERR_UNSUPPORTED;
  if (p->act_dtype == MOE_F32 && p->w_dtype == MOE_F32) {
    *path = Path::kSimt;
  } else if (p->act_dtype == MOE_BF16 && (p->w_dtype == MOE_BF16 || p->w_dtype == MOE_FP8_E4M3 ||
                                          p->w_dtype == MOE_FP8_E4M3_ACT8 || p->w_dtype == MOE_MXFP4)) {
    if (p->d % 128 != 0 || p->ffn % 128 != 0 || p->ffn_shared % 128 != 0) return MOE_ERR_UNSUPPORTED;
    *path = Path::kTensor;
  } else {
    return MOE_ERR_UNSUPPORTED;
  }
  return router_topk_check(p->d, p->E, p->act_dtype);
}

}  // namespace

moe_status problem_check(const moe_problem* p) {
  Path path;
  return check_problem(p, &path);
}

namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Largest SM count the device-free planning entry points accept.
constexpr int kMaxPlanSms = 4096;

// Quantised routed weights (FP8 or MXFP4): scale arrays required, f16 operands.
bool quantised_weights(int w_dtype) {
  return w_dtype == MOE_FP8_E4M3 || w_dtype == MOE_FP8_E4M3_ACT8 || w_dtype == MOE_MXFP4;
}

struct Layout {
  size_t idx, w, logits, counts, offsets, perm_token, inv_row, chunk, x_perm, x_scale, h, y;
  size_t sh_offsets, sh_h, sh_y, gu_part, sh_gu_part, gu_cnt, sh_gu_cnt, h_q, h_scale, total;
  size_t cnt_ints;  // gate/up finalize counters (routed, then shared), zeroed by the permutation
  size_t cnt_routed;
  TcPlan plan, sh_plan;
  int router_splits;  // 0: CUDA-core router; else tensor-core logits with this many K splits
  bool gather;        // gate/up gathers token rows (decode tiling) instead of x_perm
  bool x2_scattered;  // two-term rows written in permuted order (gate/up loads tiles)
};

// Workspace of moe_layer_forward (a superset of what the other entry points
// need).  `splits` may be forced to 1 (standalone grouped entry point).
Layout layout(const moe_problem& p, Path path, int num_sms, bool allow_splits) {
  Layout L{};
  const size_t T = p.T, k = p.k, E = p.E, R = T * k, d = p.d, f = p.ffn, ab = act_bytes(p.act_dtype);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + (bytes ? bytes : 1));
    return o;
  };
  if (path == Path::kTensor) {
    L.plan = tc_plan(p.T, p.k, p.E, p.d, p.ffn, num_sms, p.w_dtype);
    if (!allow_splits) L.plan.splits_down = L.plan.splits_gateup = 1;
    if (p.ffn_shared) {
      L.sh_plan = tc_plan(p.T, 1, 1, p.d, p.ffn_shared, num_sms, MOE_BF16);
      L.sh_plan.splits_down = 1;
    }
  }
  L.idx = take(R * 4);
  L.w = take(R * 4);
  L.router_splits = router_tc_splits(p.T, p.d, p.E, p.act_dtype, num_sms, (size_t)-1);
  L.logits = take((L.router_splits > 1 ? (size_t)L.router_splits : 1) * T * E * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.perm_token = take(R * 4);
  L.inv_row = take(R * 4);
  L.chunk = take(permute_scratch_bytes(p.T, p.k, p.E));
  // The permuted rows, except on the tensor path: there the gate/up GEMM
  // gathers the token rows itself (TMA gather4 for 32-row tiles, cp.async
  // for larger ones) and this region holds only x's two-term E4M3 rows
  // (FP8 weights: per token, or at prefill tiles scattered into the
  // permuted order, which the GEMM then loads by TMA tiles), the f16 copy
  // of x (MXFP4 weights, or FP8 weights on the converters), or x's E4M3
  // codes with FP8 activations; x_scale holds the row scales of the E4M3
  // rows.
  const bool gather = path == Path::kTensor;
  const bool act8 = p.w_dtype == MOE_FP8_E4M3_ACT8;
  const bool x2 = fp8_two_term(p.w_dtype);
  L.gather = gather;
  L.x2_scattered = gather && fp8_two_term_scattered(p.w_dtype, L.plan);
  const size_t x2_rows = L.x2_scattered ? R : T;
  const bool f16x = (p.w_dtype == MOE_FP8_E4M3 && !x2) || p.w_dtype == MOE_MXFP4;
  L.x_perm = take(gather ? (f16x ? T * d * 2 : act8 ? T * d : x2 ? 2 * x2_rows * d : 0) : R * d * ab);
  L.x_scale = take(act8 ? T * 4 : x2 ? x2_rows * 4 : 0);
  L.h = take(R * f * ab);
  // E4M3 rows of h (one per row with FP8 activations, two with two-term
  // rows) and their row scales, for the down GEMM
  L.h_q = take(act8 ? R * f : x2 ? 2 * R * f : 0);
  L.h_scale = take(act8 || x2 ? R * 4 : 0);
  const size_t S = path == Path::kTensor ? (size_t)L.plan.splits_down : 1;
  L.y = take(S > 1 ? S * R * d * 4 : R * d * ab);
  L.sh_offsets = take(8);
  L.sh_h = take(T * (size_t)p.ffn_shared * ab);
  L.sh_y = take(p.ffn_shared ? T * d * ab : 0);
  const size_t sgu = path == Path::kTensor && L.plan.splits_gateup > 1 ? L.plan.splits_gateup : 0;
  L.gu_part = take(sgu * R * 2 * f * 4);
  const size_t ssh = path == Path::kTensor && p.ffn_shared && L.sh_plan.splits_gateup > 1 ? L.sh_plan.splits_gateup : 0;
  L.sh_gu_part = take(ssh * T * 2 * (size_t)p.ffn_shared * 4);
  // arrival counters of the fused gate/up finalize (one region, zeroed by
  // the permutation of each call)
  // (decode tiles only: the finalizing warp walks the tile's rows itself)
  const size_t cr = sgu && L.plan.bn_gateup == 32 ? gu_counters_size(p.T * p.k, p.E, p.ffn, L.plan) : 0;
  const size_t cs = 0;  // (the shared expert's gate/up finalizes in its own pass)
  L.gu_cnt = take((cr + cs) * 4);
  L.sh_gu_cnt = L.gu_cnt + cr * 4;
  L.cnt_ints = cr + cs;
  L.cnt_routed = cr;
  L.total = off;
  return L;
}

bool fuse_topk_in_permute(int T, int k, int E, int router_splits) {
  return router_splits == 0 && T <= 16 && router_topk_separate(T, E, false, true) &&
         (long long)T * k <= permute_small_max();
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

__global__ void set_pair_kernel(int32_t* p, int a, int b) {
  griddep_begin();
  p[0] = a;
  p[1] = b;
}

long long wait_limit_ns() {
  static long long v = [] {
    const char* s = getenv("MOE_WAIT_LIMIT_NS");
    const long long x = s ? atoll(s) : 0;
    return x > 0 ? x : kDefaultWaitNs;
  }();
  return v;
}

// Grouped SwiGLU over `G` groups of rows, dispatched by path.
moe_status run_grouped(Path path, int R, int d, int ffn, int G, int w_dtype, const void* x_rows,
                       const int32_t* offsets, const void* wg, const void* wu, const void* wd,
                       const float* sg, const float* su, const float* sd, void* h, void* y,
                       const TcPlan& plan, int* status, cudaStream_t s, cudaEvent_t mid,
                       const int32_t* gather_rows = nullptr, const void* x_src = nullptr,
                       int T_src = 0, float* gu_partials = nullptr, int* gu_cnt = nullptr,
                       const float* row_scale = nullptr, void* h_q = nullptr, float* h_scale = nullptr,
                       int early_down = 0) {
  if (path == Path::kSimt) {
    SimtGroupedArgs a{R, d, ffn, G, static_cast<const float*>(x_rows), offsets,
                      static_cast<const float*>(wg), static_cast<const float*>(wu),
                      static_cast<const float*>(wd), static_cast<float*>(h), static_cast<float*>(y),
                      status};
    return simt_grouped_launch(a, s, mid);
  }
  TcGroupedArgs a{R, d, ffn, G, w_dtype, x_rows, offsets, wg, wu, wd, sg, su, sd, h, y, status,
                  wait_limit_ns(), gather_rows, x_src, T_src, gu_partials, gu_cnt, row_scale, h_q, h_scale,
                  early_down};
  return tc_grouped_launch(a, plan, s, mid);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_workspace_size_for(const moe_problem* p, int32_t num_sms, size_t* bytes) {
  if (bytes == nullptr || num_sms < 1 || num_sms > kMaxPlanSms) return MOE_ERR_INVALID_ARG;
  Path path;
  MOE_TRY(check_problem(p, &path));
  *bytes = layout(*p, path, num_sms, true).total;
  return MOE_OK;
}

moe_status moe_workspace_size(const moe_problem* p, size_t* bytes) {
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  Path path;
  MOE_TRY(check_problem(p, &path));
  DeviceCtx ctx;
  MOE_TRY(device_ctx(&ctx));
  return moe_workspace_size_for(p, ctx.num_sms, bytes);
}

moe_status moe_router_topk(const moe_problem* p, const void* x, const void* w_router,
                           const float* router_bias, const float* logits_in, float* logits_out,
                           int32_t* topk_idx, float* topk_w, moe_stream_t stream) {
  Path path;
  MOE_TRY(check_problem(p, &path));
  if (topk_idx == nullptr || topk_w == nullptr) return MOE_ERR_INVALID_ARG;
  if (logits_in != nullptr && router_bias != nullptr) return MOE_ERR_INVALID_ARG;
  if (logits_in == nullptr && (x == nullptr || w_router == nullptr)) return MOE_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || (w_router && !aligned16(w_router))) return MOE_ERR_INVALID_ARG;
  if (p->T == 0) return MOE_OK;
  DeviceCtx ctx;
  MOE_TRY(device_ctx(&ctx));
  // tensor-core logits need a global buffer: only when the caller gave one
  const int tcs = logits_out ? router_tc_splits(p->T, p->d, p->E, p->act_dtype, ctx.num_sms,
                                                (size_t)p->T * p->E)
                             : 0;
  RouterArgs a{p->T, p->d, p->E, p->k, p->act_dtype, x, w_router, router_bias, logits_in,
               logits_out, topk_idx, topk_w, logits_out, tcs, ctx.num_sms, ctx.status};
  return router_topk_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_permute(const moe_problem* p, const int32_t* topk_idx, const void* x,
                       int32_t* counts, int32_t* offsets, int32_t* perm_token, int32_t* inv_row,
                       void* x_perm, void* workspace, size_t workspace_bytes,
                       moe_stream_t stream) {
  Path path;
  MOE_TRY(check_problem(p, &path));
  if (counts == nullptr || offsets == nullptr || perm_token == nullptr || inv_row == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && topk_idx == nullptr) return MOE_ERR_INVALID_ARG;
  if ((x_perm != nullptr) != (x != nullptr)) return MOE_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || (x_perm && !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
  const size_t scratch = permute_scratch_bytes(p->T, p->k, p->E);
  if (scratch > 0 && (workspace == nullptr || workspace_bytes < scratch)) return MOE_ERR_WORKSPACE;
  DeviceCtx ctx;
  MOE_TRY(device_ctx(&ctx));
  PermuteArgs a{p->T, p->k, p->E, p->d, (int)act_bytes(p->act_dtype), topk_idx, x, counts,
                offsets, perm_token, inv_row, x_perm, static_cast<int32_t*>(workspace),
                ctx.status};
  return permute_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_grouped_swiglu(const moe_problem* p, const void* x_perm, const int32_t* offsets,
                              const void* w_gate, const void* w_up, const void* w_down,
                              const float* s_gate, const float* s_up, const float* s_down,
                              void* y_perm, void* workspace, size_t workspace_bytes,
                              moe_stream_t stream) {
  Path path;
  MOE_TRY(check_problem(p, &path));
  if (p->T == 0) return MOE_OK;
  if (!x_perm || !offsets || !w_gate || !w_up || !w_down || !y_perm) return MOE_ERR_INVALID_ARG;
  for (const void* q : {x_perm, w_gate, w_up, w_down, (const void*)y_perm})
    if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
  const bool fp8 = quantised_weights(p->w_dtype), act8 = p->w_dtype == MOE_FP8_E4M3_ACT8;
  const bool x2 = fp8_two_term(p->w_dtype);
  if (fp8 != (s_gate != nullptr) || fp8 != (s_up != nullptr) || fp8 != (s_down != nullptr))
    return MOE_ERR_INVALID_ARG;
  DeviceCtx ctx;
  MOE_TRY(device_ctx(&ctx));
  const Layout L = layout(*p, path, ctx.num_sms, false);
  const size_t R = (size_t)p->T * p->k;
  const size_t h_bytes = align256(R * p->ffn * act_bytes(p->act_dtype));
  // FP8 weights: x_perm's rows split into two E4M3 rows each (or, on the
  // converters, rounded to f16); with FP8 activations, their E4M3 codes;
  // E4M3 rows come with row scales
  const size_t rows_bytes = act8 ? align256(R * p->d) : x2 ? align256(2 * R * p->d)
                                                       : fp8 ? align256(R * p->d * 2) : 0;
  const bool e4m3_rows = act8 || x2;
  // (E4M3 rows: x_perm's codes, their scales, then h's codes and scales)
  const size_t hq_off = h_bytes + rows_bytes + (e4m3_rows ? align256(R * 4) : 0);
  const size_t hq_bytes = act8 ? align256(R * p->ffn) : x2 ? align256(2 * R * p->ffn) : 0;
  const size_t need = hq_off + (e4m3_rows ? hq_bytes + align256(R * 4) : 0);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const void* rows = x_perm;
  float* row_scale = nullptr;
  if (e4m3_rows) {
    row_scale = at<float>(workspace, h_bytes + rows_bytes);
    if (x2)
      MOE_TRY(split_rows_e4m3x2_launch(x_perm, (int)R, p->d, at<uint8_t>(workspace, h_bytes), row_scale,
                                       ctx.num_sms, s));
    else
      MOE_TRY(quantize_rows_e4m3_launch(x_perm, (int)R, p->d, at<uint8_t>(workspace, h_bytes), row_scale,
                                        ctx.num_sms, s));
    rows = at<uint8_t>(workspace, h_bytes);
  } else if (fp8) {
    void* xf16 = at<uint8_t>(workspace, h_bytes);
    MOE_TRY(bf16_to_f16_launch(x_perm, xf16, R * p->d, s));
    rows = xf16;
  }
  return run_grouped(path, (int)R, p->d, p->ffn, p->E, p->w_dtype, rows, offsets, w_gate, w_up,
                     w_down, s_gate, s_up, s_down, workspace, y_perm, L.plan, ctx.status, s,
                     nullptr, nullptr, nullptr, 0, nullptr, nullptr, row_scale,
                     e4m3_rows ? at<uint8_t>(workspace, hq_off) : nullptr,
                     e4m3_rows ? at<float>(workspace, hq_off + hq_bytes) : nullptr);
}

moe_status moe_quantize_rows_e4m3(int32_t rows, int32_t cols, const void* x, uint8_t* codes,
                                  float* scales, moe_stream_t stream) {
  if (rows < 0) return MOE_ERR_INVALID_ARG;
  if (cols <= 0 || cols % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  if (x == nullptr || codes == nullptr || scales == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0)
    return MOE_ERR_INVALID_ARG;
  DeviceCtx ctx;
  MOE_TRY(device_ctx(&ctx));
  return quantize_rows_e4m3_launch(x, rows, cols, codes, scales, ctx.num_sms,
                                   reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_split_rows_e4m3x2(int32_t rows, int32_t cols, const void* x, uint8_t* codes, float* scales,
                                 moe_stream_t stream) {
  if (rows < 0) return MOE_ERR_INVALID_ARG;
  if (cols <= 0 || cols % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  if (x == nullptr || codes == nullptr || scales == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0)
    return MOE_ERR_INVALID_ARG;
  DeviceCtx ctx;
  MOE_TRY(device_ctx(&ctx));
  return split_rows_e4m3x2_launch(x, rows, cols, codes, scales, ctx.num_sms,
                                  reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_combine(const moe_problem* p, const void* y_perm, const int32_t* inv_row,
                       const float* topk_w, const void* shared_out, void* out,
                       moe_stream_t stream) {
  Path path;
  MOE_TRY(check_problem(p, &path));
  if (p->T == 0) return MOE_OK;
  if (!y_perm || !inv_row || !topk_w || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(out) || (shared_out && !aligned16(shared_out)))
    return MOE_ERR_INVALID_ARG;
  CombineArgs a{p->T, p->k, p->d, p->act_dtype, y_perm, 0, inv_row, topk_w, shared_out, out};
  return combine_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

struct moe_stage_timer {
  cudaEvent_t ev[MOE_NUM_STAGES + 1];
  int recorded;
};

namespace moe {
namespace {

moe_status layer_forward_impl(const moe_problem* p, const void* x, const void* w_router,
                              const float* router_bias, const void* w_gate, const void* w_up,
                              const void* w_down, const float* s_gate, const float* s_up,
                              const float* s_down, const void* w_shared_gate,
                              const void* w_shared_up, const void* w_shared_down, void* out,
                              int32_t* topk_idx_out, float* topk_w_out, int32_t* counts_out,
                              void* workspace, size_t workspace_bytes, moe_stream_t stream,
                              moe_stage_timer* timer) {
  Path path;
  MOE_TRY(check_problem(p, &path));
  if (p->T == 0) return MOE_OK;
  if (!x || !w_router || !w_gate || !w_up || !w_down || !out) return MOE_ERR_INVALID_ARG;
  for (const void* q : {x, w_router, w_gate, w_up, w_down, (const void*)out})
    if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
  const bool fp8 = quantised_weights(p->w_dtype), act8 = p->w_dtype == MOE_FP8_E4M3_ACT8;
  if (fp8 != (s_gate != nullptr) || fp8 != (s_up != nullptr) || fp8 != (s_down != nullptr))
    return MOE_ERR_INVALID_ARG;
  const bool has_shared = p->ffn_shared > 0;
  if (has_shared != (w_shared_gate != nullptr) || has_shared != (w_shared_up != nullptr) ||
      has_shared != (w_shared_down != nullptr))
    return MOE_ERR_INVALID_ARG;
  if (has_shared && (!aligned16(w_shared_gate) || !aligned16(w_shared_up) || !aligned16(w_shared_down)))
    return MOE_ERR_INVALID_ARG;
  DeviceCtx ctx;
  MOE_TRY(device_ctx(&ctx));
  const Layout L = layout(*p, path, ctx.num_sms, true);
  if (workspace == nullptr || workspace_bytes < L.total || !aligned16(workspace))
    return MOE_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int R = p->T * p->k;
  auto mark = [&](int i) -> moe_status {
    if (timer != nullptr) {
      MOE_TRY_CUDA(record_event(timer->ev[i], s));
      timer->recorded = i + 1;
    }
    return MOE_OK;
  };

  int32_t* idx = topk_idx_out ? topk_idx_out : at<int32_t>(workspace, L.idx);
  float* w = topk_w_out ? topk_w_out : at<float>(workspace, L.w);
  int32_t* counts = counts_out ? counts_out : at<int32_t>(workspace, L.counts);
  int32_t* offsets = at<int32_t>(workspace, L.offsets);
  int32_t* perm_token = at<int32_t>(workspace, L.perm_token);
  int32_t* inv_row = at<int32_t>(workspace, L.inv_row);
  void* x_perm = at<uint8_t>(workspace, L.x_perm);
  void* h = at<uint8_t>(workspace, L.h);
  void* y = at<uint8_t>(workspace, L.y);

  MOE_TRY(mark(0));
  // 4. (first) shared expert: every token, weight 1.  On the tensor path it
  // needs only x, so it runs on the side stream, concurrently with routing
  // and permutation (whose small kernels share the SMs with it); the
  // combine joins it.  Its split-K gate/up finalizes in a separate pass.
  void* sh_y = nullptr;
  const bool side = has_shared && path == Path::kTensor;
  if (side) {
    sh_y = at<uint8_t>(workspace, L.sh_y);
    MOE_TRY_CUDA(cudaEventRecord(ctx.fork, s));
    MOE_TRY_CUDA(cudaStreamWaitEvent(ctx.side, ctx.fork, 0));
    MOE_TRY(run_grouped(path, p->T, p->d, p->ffn_shared, 1, p->act_dtype, x, nullptr, w_shared_gate,
                        w_shared_up, w_shared_down, nullptr, nullptr, nullptr, at<uint8_t>(workspace, L.sh_h),
                        sh_y, L.sh_plan, ctx.status, ctx.side, nullptr, nullptr, nullptr, 0,
                        at<float>(workspace, L.sh_gu_part), nullptr));
    MOE_TRY_CUDA(cudaEventRecord(ctx.join, ctx.side));
  }
  // 1. router: logits, softmax, top-k, renormalised weights
  // the logits region is the CUDA-core split path's buffer, or the tensor
  // core's partial-sum scratch (the logits themselves are not an output here)
  float* lg = at<float>(workspace, L.logits);
  // tiny batches (a token per warp of the one-block permutation): the
  // permutation kernel selects the top-k from the global logits itself
  // (one launch fewer on the latency-bound path)
  const bool fuse_topk = fuse_topk_in_permute(p->T, p->k, p->E, L.router_splits);
  RouterArgs ra{p->T, p->d, p->E, p->k, p->act_dtype, x, w_router, router_bias, nullptr,
                L.router_splits > 0 ? nullptr : lg, idx, w, lg, L.router_splits, ctx.num_sms,
                ctx.status, fuse_topk ? 1 : 0};
  MOE_TRY(router_topk_launch(ra, s));
  MOE_TRY(mark(1));
  // 2. permutation: counts, offsets, row maps, x -> x_perm
  // On the tensor path the permutation writes only the maps: the gate/up
  // GEMM gathers token rows by perm_token itself (FP8 experts gather from an
  // f16 copy of x).  On the CUDA-core path the row move fills x_perm.
  const bool gather = L.gather;
  PermuteArgs pa{p->T, p->k, p->E, p->d, (int)act_bytes(p->act_dtype), idx, gather ? nullptr : x,
                 counts, offsets, perm_token, inv_row, gather ? nullptr : x_perm,
                 at<int32_t>(workspace, L.chunk), ctx.status, fp8 && !gather ? 1 : 0,
                 fuse_topk ? lg : nullptr, fuse_topk ? idx : nullptr, fuse_topk ? w : nullptr,
                 L.cnt_ints ? at<int32_t>(workspace, L.gu_cnt) : nullptr, L.cnt_ints};
  MOE_TRY(permute_launch(pa, s));
  MOE_TRY(mark(2));
  // 3. grouped SwiGLU experts (gate/up + SiLU*mul, then down)
  // FP8 experts gather from an f16 copy of x; with FP8 activations, from
  // x's per-row E4M3 codes (quantised before dispatch: T rows, not T*k)
  // FP8 weights gather x's two-term E4M3 rows (split once per token, before
  // dispatch)
  const void* x_src = x;
  float* x_scale = nullptr;
  const bool x2 = fp8_two_term(p->w_dtype);
  if (gather && act8) {
    x_scale = at<float>(workspace, L.x_scale);
    MOE_TRY(quantize_rows_e4m3_launch(x, p->T, p->d, x_perm, x_scale, ctx.num_sms, s));
    x_src = x_perm;
  } else if (gather && x2 && L.x2_scattered) {
    // prefill tiles: each token's two rows written to its k permuted rows
    // (tile loads in the GEMM instead of a two-row gather per row)
    x_scale = at<float>(workspace, L.x_scale);
    MOE_TRY(split_rows_e4m3x2_scatter_launch(x, p->T, p->d, p->k, inv_row, R, x_perm, x_scale, ctx.status,
                                             ctx.num_sms, s));
  } else if (gather && x2) {
    x_scale = at<float>(workspace, L.x_scale);
    MOE_TRY(split_rows_e4m3x2_launch(x, p->T, p->d, x_perm, x_scale, ctx.num_sms, s));
    x_src = x_perm;
  } else if (gather && fp8) {
    MOE_TRY(bf16_to_f16_launch(x, x_perm, (size_t)p->T * p->d, s));
    x_src = x_perm;
  }
  const bool gathered = gather && !L.x2_scattered;
  MOE_TRY(run_grouped(path, R, p->d, p->ffn, p->E, p->w_dtype, x_perm, offsets, w_gate, w_up,
                      w_down, s_gate, s_up, s_down, h, y, L.plan, ctx.status, s,
                      timer ? timer->ev[3] : nullptr, gathered ? perm_token : nullptr, x_src, p->T,
                      at<float>(workspace, L.gu_part), L.cnt_routed ? at<int>(workspace, L.gu_cnt) : nullptr,
                      x_scale, act8 || x2 ? at<uint8_t>(workspace, L.h_q) : nullptr,
                      act8 || x2 ? at<float>(workspace, L.h_scale) : nullptr,
                      /* early_down: the permutation above wrote the offsets */ 1));
  MOE_TRY(mark(4));
  // 4. shared expert (CUDA-core path: here, one group {0, T}); on the
  // tensor path, join the side stream
  if (side) {
    MOE_TRY_CUDA(cudaStreamWaitEvent(s, ctx.join, 0));
  } else if (has_shared) {
    int32_t* sh_off = at<int32_t>(workspace, L.sh_offsets);
    MOE_TRY_CUDA(launch_k(set_pair_kernel, dim3(1), dim3(1), 0, s, sh_off, 0, p->T));
    MOE_TRY_CUDA(cudaGetLastError());
    sh_y = at<uint8_t>(workspace, L.sh_y);
    MOE_TRY(run_grouped(path, p->T, p->d, p->ffn_shared, 1, p->act_dtype, x, sh_off,
                        w_shared_gate, w_shared_up, w_shared_down, nullptr, nullptr, nullptr,
                        at<uint8_t>(workspace, L.sh_h), sh_y, L.sh_plan, ctx.status, s, nullptr,
                        nullptr, nullptr, 0, at<float>(workspace, L.sh_gu_part), nullptr));
  }
  MOE_TRY(mark(5));
  // 5. combine: inverse map, routing weights, sum (+ shared expert)
  const int partials = path == Path::kTensor && L.plan.splits_down > 1 ? L.plan.splits_down : 0;
  CombineArgs ca{p->T, p->k, p->d, p->act_dtype, y, partials, inv_row, w, sh_y, out};
  MOE_TRY(combine_launch(ca, s));
  return mark(6);
}

}  // namespace
}  // namespace moe

extern "C" {

moe_status moe_layer_forward(const moe_problem* p, const void* x, const void* w_router,
                             const float* router_bias, const void* w_gate, const void* w_up,
                             const void* w_down, const float* s_gate, const float* s_up,
                             const float* s_down, const void* w_shared_gate,
                             const void* w_shared_up, const void* w_shared_down, void* out,
                             int32_t* topk_idx_out, float* topk_w_out, int32_t* counts_out,
                             void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  return layer_forward_impl(p, x, w_router, router_bias, w_gate, w_up, w_down, s_gate, s_up,
                            s_down, w_shared_gate, w_shared_up, w_shared_down, out, topk_idx_out,
                            topk_w_out, counts_out, workspace, workspace_bytes, stream, nullptr);
}

moe_status moe_layer_forward_timed(const moe_problem* p, const void* x, const void* w_router,
                                   const float* router_bias, const void* w_gate, const void* w_up,
                                   const void* w_down, const float* s_gate, const float* s_up,
                                   const float* s_down, const void* w_shared_gate,
                                   const void* w_shared_up, const void* w_shared_down, void* out,
                                   int32_t* topk_idx_out, float* topk_w_out, int32_t* counts_out,
                                   void* workspace, size_t workspace_bytes, moe_stream_t stream,
                                   moe_stage_timer* timer) {
  if (timer == nullptr) return MOE_ERR_INVALID_ARG;
  timer->recorded = 0;
  return layer_forward_impl(p, x, w_router, router_bias, w_gate, w_up, w_down, s_gate, s_up,
                            s_down, w_shared_gate, w_shared_up, w_shared_down, out, topk_idx_out,
                            topk_w_out, counts_out, workspace, workspace_bytes, stream, timer);
}

moe_status moe_stage_timer_create(moe_stage_timer** timer) {
  if (timer == nullptr) return MOE_ERR_INVALID_ARG;
  moe_stage_timer* t = new moe_stage_timer();
  for (int i = 0; i <= MOE_NUM_STAGES; ++i) {
    cudaError_t e = cudaEventCreate(&t->ev[i]);
    if (e != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(t->ev[j]);
      delete t;
      return cuda_status(e);
    }
  }
  t->recorded = 0;
  *timer = t;
  return MOE_OK;
}

moe_status moe_stage_timer_destroy(moe_stage_timer* timer) {
  if (timer == nullptr) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i <= MOE_NUM_STAGES; ++i) cudaEventDestroy(timer->ev[i]);
  delete timer;
  return MOE_OK;
}

moe_status moe_stage_timer_read(moe_stage_timer* timer, float* ms) {
  if (timer == nullptr || ms == nullptr) return MOE_ERR_INVALID_ARG;
  if (timer->recorded != MOE_NUM_STAGES + 1) return MOE_ERR_INVALID_ARG;
  MOE_TRY_CUDA(cudaEventSynchronize(timer->ev[MOE_NUM_STAGES]));
  for (int i = 0; i < MOE_NUM_STAGES; ++i)
    MOE_TRY_CUDA(cudaEventElapsedTime(&ms[i], timer->ev[i], timer->ev[i + 1]));
  return MOE_OK;
}

moe_status moe_plan_info(const moe_problem* p, int32_t* info) {
  if (info == nullptr) return MOE_ERR_INVALID_ARG;
  Path path;
  MOE_TRY(check_problem(p, &path));
  if (path != Path::kTensor) {  // the CUDA-core path has no tiling to report
    info[0] = info[1] = info[2] = info[3] = info[4] = info[5] = 0;
    return MOE_OK;
  }
  DeviceCtx ctx;
  MOE_TRY(device_ctx(&ctx));
  return moe_plan_info_for(p, ctx.num_sms, info);
}

moe_status moe_plan_info_for(const moe_problem* p, int32_t num_sms, int32_t* info) {
  if (info == nullptr || num_sms < 1 || num_sms > kMaxPlanSms) return MOE_ERR_INVALID_ARG;
  Path path;
  MOE_TRY(check_problem(p, &path));
  info[0] = info[1] = info[2] = info[3] = info[4] = info[5] = 0;
  if (path != Path::kTensor) return MOE_OK;
  const Layout L = layout(*p, path, num_sms, true);
  info[0] = L.plan.bn_gateup;
  info[1] = L.plan.bn_down;
  info[2] = L.plan.splits_down;
  info[3] = L.plan.grid;
  info[4] = L.plan.splits_gateup;
  info[5] = (L.plan.pair_gateup ? 1 : 0) | (L.plan.pair_down ? 2 : 0);
  return MOE_OK;
}

moe_status moe_layer_launch_count(const moe_problem* p, int32_t* launches) {
  if (launches == nullptr) return MOE_ERR_INVALID_ARG;
  Path path;
  MOE_TRY(check_problem(p, &path));
  if (p->T == 0) {
    *launches = 0;
    return MOE_OK;
  }
  DeviceCtx ctx;
  MOE_TRY(device_ctx(&ctx));
  return moe_layer_launch_count_for(p, ctx.num_sms, launches);
}

moe_status moe_layer_launch_count_for(const moe_problem* p, int32_t num_sms, int32_t* launches) {
  if (launches == nullptr || num_sms < 1 || num_sms > kMaxPlanSms) return MOE_ERR_INVALID_ARG;
  Path path;
  MOE_TRY(check_problem(p, &path));
  if (p->T == 0) {
    *launches = 0;
    return MOE_OK;
  }
  const int rs = router_tc_splits(p->T, p->d, p->E, p->act_dtype, num_sms, (size_t)-1);
  int n = rs > 0 ? 2 : router_launch_count(p->T, p->E, false, true);
  // the tiny-batch permutation selects the top-k in place of the separate pass
  if (fuse_topk_in_permute(p->T, p->k, p->E, rs)) n -= 1;
  const Layout L = layout(*p, path, num_sms, true);
  n += permute_launch_count(p->T, p->k, !L.gather);
  if (L.gather && quantised_weights(p->w_dtype)) n += 1;  // x -> f16, or x -> E4M3 rows
  // h -> E4M3 codes, or h -> two-term E4M3 rows
  if (p->w_dtype == MOE_FP8_E4M3_ACT8 || (path == Path::kTensor && fp8_two_term(p->w_dtype))) n += 1;
  n += 2;                        // gate/up, down
  // split-K gate/up: a finalize pass unless the GEMM finalizes itself
  // (decode tiles)
  if (path == Path::kTensor && L.plan.splits_gateup > 1 && L.plan.bn_gateup != 32) n += 1;
  if (path == Path::kTensor && p->ffn_shared > 0 && L.sh_plan.splits_gateup > 1) n += 1;
  if (p->ffn_shared > 0) n += path == Path::kTensor ? 2 : 3;  // (offsets), gate/up, down
  n += 1;                        // combine
  *launches = n;
  return MOE_OK;
}

moe_status moe_selftest_bounded_wait(int64_t timeout_ns, moe_stream_t stream) {
  if (timeout_ns <= 0) return MOE_ERR_INVALID_ARG;
  DeviceCtx ctx;
  MOE_TRY(device_ctx(&ctx));
  return tc_selftest_launch(ctx.status, timeout_ns, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
