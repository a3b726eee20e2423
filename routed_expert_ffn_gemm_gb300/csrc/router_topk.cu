// Router: logits l = x W_r^T (+ b) in fp32, then softmax / top-k /
// renormalisation per token ("MOE推理流程解析", section 三: the router
// scores every eligible expert, top-k keeps the chosen indices and weights;
// section 九: the kept weights are re-normalised).
//
// router_kernel: a block owns TT tokens (8, or 1 for small batches), whose
// rows are staged once in shared memory, and a slice of the experts; each
// warp accumulates EPW experts x TT tokens with 16-byte loads of W_r rows
// (fp32 FMA, the hidden loop unrolled so several loads are in flight) and a
// shuffle reduction.  With one expert slice (gridDim.y == 1, "fused") the logits stay
// in shared memory and the same block selects the top-k; with several slices
// (few tokens: more blocks stream W_r) the logits go to global memory and
// topk_kernel follows (or, at small batches inside the layer, the
// permutation kernel selects the top-k itself).  Selection and weights:
// topk_row (topk.cuh).
#include "common.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kTT = 8;  // tokens per block (large batches)
// Batches from 256 tokens take the tensor-core logits (E % 128 == 0, bf16),
// and from 32 when W_r is large (d*E >= 2^20): the W_r tiles stream through
// TMA into tcgen05 with the K range split over the SMs, where the CUDA-core
// kernel re-reads W_r per 8-token tile.  Below that the CUDA-core kernels'
// two short launches measured faster on GB300.
bool tc_router_size(int T, int d, int E) { return T >= 256 || (T >= 32 && (long long)d * E >= (1LL << 20)); }
constexpr int kThreads = 256;

__device__ __forceinline__ void load16(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void load16(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&a);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
template <typename T> struct VecN { static constexpr int N = 16 / sizeof(T); };

template <typename ActT, int EPW, int TT>
__global__ void __launch_bounds__(kThreads) router_kernel(
    int T, int d, int E, int k, const ActT* __restrict__ x, const ActT* __restrict__ wr,
    const float* __restrict__ bias, const float* __restrict__ logits_in,
    float* __restrict__ logits_out, int32_t* __restrict__ idx, float* __restrict__ w) {
  griddep_begin();
  constexpr int VN = VecN<ActT>::N;
  extern __shared__ __align__(16) uint8_t sm[];
  const bool fused = gridDim.y == 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * TT;
  ActT* xs = reinterpret_cast<ActT*>(sm);                                   // [TT][d]
  float* ls = reinterpret_cast<float*>(sm + (logits_in ? 0 : sizeof(ActT) * TT * d));  // [TT][E]

  if (logits_in == nullptr) {
    const int vec_per_row = d / VN;
#pragma unroll 4
    for (int v = threadIdx.x; v < TT * vec_per_row; v += kThreads) {
      const int t = v / vec_per_row, c = (v % vec_per_row) * VN;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (t0 + t < T) val = *reinterpret_cast<const uint4*>(x + (size_t)(t0 + t) * d + c);
      *reinterpret_cast<uint4*>(xs + (size_t)t * d + c) = val;
    }
    __syncthreads();
    const int slice = ((E + gridDim.y - 1) / gridDim.y + EPW - 1) / EPW * EPW;
    const int e_lo = blockIdx.y * slice, e_hi = min(E, e_lo + slice);
    for (int eb = e_lo + warp * EPW; eb < e_hi; eb += 8 * EPW) {
      float acc[EPW][TT];
#pragma unroll
      for (int a = 0; a < EPW; ++a)
#pragma unroll
        for (int t = 0; t < TT; ++t) acc[a][t] = 0.f;
#pragma unroll 8
      for (int i = lane * VN; i < d; i += 32 * VN) {
        float xv[TT][8];
#pragma unroll
        for (int t = 0; t < TT; ++t) load16(xs + (size_t)t * d + i, xv[t]);
#pragma unroll
        for (int a = 0; a < EPW; ++a) {
          if (eb + a < e_hi) {
            float wv[8];
            load16(wr + (size_t)(eb + a) * d + i, wv);
#pragma unroll
            for (int t = 0; t < TT; ++t)
#pragma unroll
              for (int q = 0; q < VN; ++q) acc[a][t] = fmaf(wv[q], xv[t][q], acc[a][t]);
          }
        }
      }
#pragma unroll
      for (int a = 0; a < EPW; ++a) {
        const int e = eb + a;
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          float v = acc[a][t];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0 && e < e_hi) {
            v += bias != nullptr ? bias[e] : 0.f;
            if (fused) ls[t * E + e] = v;
            if (logits_out != nullptr && t0 + t < T) logits_out[(size_t)(t0 + t) * E + e] = v;
          }
        }
      }
    }
  } else {
    for (int i = threadIdx.x; i < TT * E; i += kThreads) {
      const int t = i / E;
      ls[i] = t0 + t < T ? logits_in[(size_t)t0 * E + i] : 0.f;
    }
  }
  if (!fused) return;
  __syncthreads();
  // one warp per token
  for (int t = warp; t < TT; t += kThreads / 32)
    if (t0 + t < T) topk_row(ls + t * E, E, k, idx + (size_t)(t0 + t) * k, w + (size_t)(t0 + t) * k);
}

// One warp per token; the row is staged in shared memory once (the k
// selection rounds read it k times).
__global__ void __launch_bounds__(kThreads) topk_kernel(int T, int E, int k,
                                                        const float* __restrict__ logits,
                                                        int32_t* __restrict__ idx,
                                                        float* __restrict__ w) {
  griddep_begin();
  extern __shared__ float rows[];  // [8][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kThreads / 32) + warp;
  if (t >= T) return;
  float* row = rows + warp * E;
  for (int e = lane; e < E; e += 32) row[e] = logits[(size_t)t * E + e];
  __syncwarp();
  topk_row(row, E, k, idx + (size_t)t * k, w + (size_t)t * k);
}

// Top-k after the tensor-core logits: l[t, :] = sum_s part[s][t][:] (s in
// order) + bias, staged per warp in shared memory (optionally written out).
__global__ void __launch_bounds__(kThreads) topk_partials_kernel(
    int T, int E, int k, int S, const float* __restrict__ part, const float* __restrict__ bias,
    float* __restrict__ logits_out, int32_t* __restrict__ idx, float* __restrict__ w) {
  griddep_begin();
  extern __shared__ float rows[];  // [8][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kThreads / 32) + warp;
  if (t >= T) return;
  float* row = rows + warp * E;
  for (int e = lane; e < E; e += 32) {
    float v = part[(size_t)t * E + e];
    for (int s = 1; s < S; ++s) v += part[((size_t)s * T + t) * E + e];
    if (bias != nullptr) v += bias[e];
    row[e] = v;
    if (logits_out != nullptr) logits_out[(size_t)t * E + e] = v;
  }
  __syncwarp();
  topk_row(row, E, k, idx + (size_t)t * k, w + (size_t)t * k);
}

// Few tokens and a global logits buffer available: split the experts over
// more blocks (one expert per warp, one token per block when the batch is
// tiny), then a separate top-k pass unless one block sees all experts.
bool use_split(int T, int E, bool logits_in, bool scratch) {
  return !logits_in && scratch && T <= 512;
}
int split_tt(int T) { return T <= 128 ? 1 : kTT; }
bool split_needs_topk_pass(int E) { return (E + 7) / 8 > 1; }

template <typename ActT>
moe_status launch_typed(const RouterArgs& a, float* logits_scratch, cudaStream_t s) {
  const bool split = use_split(a.T, a.E, a.logits_in != nullptr, logits_scratch != nullptr);
  if (split) {
    const int tt = split_tt(a.T);
    const size_t xs_bytes = sizeof(ActT) * tt * a.d;
    const int gy = (a.E + 7) / 8;
    // one block row sees every expert: keep the logits in shared memory
    const size_t smem = xs_bytes + (gy == 1 ? sizeof(float) * tt * a.E : 0);
    dim3 grid((a.T + tt - 1) / tt, gy);
    if (tt == 1) {
      auto kern = router_kernel<ActT, 1, 1>;
      MOE_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
      MOE_TRY_CUDA(launch_k(kern, dim3(grid), dim3(kThreads), smem, s, a.T, a.d, a.E, a.k, static_cast<const ActT*>(a.x),
                                        static_cast<const ActT*>(a.w_router), a.bias, nullptr,
                                        logits_scratch, a.idx, a.w));
    } else {
      auto kern = router_kernel<ActT, 1, kTT>;
      MOE_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
      MOE_TRY_CUDA(launch_k(kern, dim3(grid), dim3(kThreads), smem, s, a.T, a.d, a.E, a.k, static_cast<const ActT*>(a.x),
                                        static_cast<const ActT*>(a.w_router), a.bias, nullptr,
                                        logits_scratch, a.idx, a.w));
    }
    MOE_TRY_CUDA(cudaGetLastError());
    if (gy > 1 && !a.defer_topk) {
      const size_t tsmem = sizeof(float) * 8 * a.E;
      MOE_TRY_CUDA(cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tsmem));
      MOE_TRY_CUDA(launch_k(topk_kernel, dim3((a.T + 7) / 8), dim3(kThreads), tsmem, s, a.T, a.E, a.k, logits_scratch,
                            a.idx, a.w));
      MOE_TRY_CUDA(cudaGetLastError());
    }
    return MOE_OK;
  }
  const int tiles = (a.T + kTT - 1) / kTT;
  const size_t xs_bytes = a.logits_in ? 0 : sizeof(ActT) * kTT * a.d;
  const size_t smem = xs_bytes + sizeof(float) * kTT * a.E;
  if (smem > 220 * 1024) return MOE_ERR_UNSUPPORTED;
  auto kern = router_kernel<ActT, 4, kTT>;
  MOE_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  MOE_TRY_CUDA(launch_k(kern, dim3(dim3(tiles, 1)), dim3(kThreads), smem, s, a.T, a.d, a.E, a.k, static_cast<const ActT*>(a.x),
                                              static_cast<const ActT*>(a.w_router), a.bias,
                                              a.logits_in, a.logits_out, a.idx, a.w));
  MOE_TRY_CUDA(cudaGetLastError());
  if (a.logits_in != nullptr && a.logits_out != nullptr && a.logits_out != a.logits_in)
    MOE_TRY_CUDA(cudaMemcpyAsync(a.logits_out, a.logits_in, sizeof(float) * a.T * a.E,
                                 cudaMemcpyDeviceToDevice, s));
  return MOE_OK;
}

}  // namespace

int router_launch_count(int T, int E, bool logits_in, bool logits_out) {
  return use_split(T, E, logits_in, logits_out) && split_needs_topk_pass(E) ? 2 : 1;
}

bool router_topk_separate(int T, int E, bool logits_in, bool logits_out) {
  return use_split(T, E, logits_in, logits_out) && split_needs_topk_pass(E);
}

moe_status router_topk_check(int d, int E, int act_dtype) {
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  if (act_dtype != MOE_F32 && act_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  const size_t act = act_dtype == MOE_F32 ? 4 : 2;
  if (act * kTT * d + sizeof(float) * kTT * E > 220 * 1024) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int router_tc_splits(int T, int d, int E, int act_dtype, int num_sms, size_t scratch_floats) {
  if (act_dtype != MOE_BF16 || E % 128 != 0 || !tc_router_size(T, d, E) || d % 64 != 0) return 0;
  if ((size_t)T * E > scratch_floats) return 0;
  const int tiles = ((T + 127) / 128) * (E / 128);
  const int kblocks = d / 64;
  // as many K splits as keep every unit in one wave of the SMs (a partial
  // second wave costs a whole unit's time), each split >= 8 k-blocks
  int splits = 1;
  while ((splits + 1) * tiles <= num_sms && splits < 16 && kblocks / (splits + 1) >= 8) ++splits;
  while (splits > 1 && (size_t)splits * T * E > scratch_floats) --splits;
  return splits;
}

moe_status router_topk_launch(const RouterArgs& a, cudaStream_t s) {
  if (a.T == 0) return MOE_OK;
  MOE_TRY(router_topk_check(a.d, a.E, a.act_dtype));
  if (a.logits_in == nullptr && a.tc_splits > 0 && a.tc_scratch != nullptr) {
    // logits on the tensor cores: [splits][T][E] fp32 partials
    MOE_TRY(tc_dense_f32_launch(a.w_router, a.x, a.tc_scratch, a.E, a.T, a.d, a.tc_splits,
                                a.num_sms, a.status, kDefaultWaitNs, s));
    const size_t smem = sizeof(float) * 8 * a.E;
    MOE_TRY_CUDA(cudaFuncSetAttribute(topk_partials_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    // logits_out may be the scratch itself when there is one split: each
    // element is read, then rewritten (biased) by the same lane
    float* lo = a.logits_out;
    if (lo == a.tc_scratch && a.tc_splits > 1) return MOE_ERR_INVALID_ARG;
    MOE_TRY_CUDA(launch_k(topk_partials_kernel, dim3((a.T + 7) / 8), dim3(kThreads), smem, s, a.T, a.E, a.k, a.tc_splits, a.tc_scratch,
                                                               a.bias, lo, a.idx, a.w));
    MOE_TRY_CUDA(cudaGetLastError());
    return MOE_OK;
  }
  // a caller-visible logits_out doubles as the split path's global buffer
  float* scratch = a.logits_out;
  if (a.act_dtype == MOE_BF16) return launch_typed<__nv_bfloat16>(a, scratch, s);
  return launch_typed<float>(a, scratch, s);
}

}  // namespace moe
