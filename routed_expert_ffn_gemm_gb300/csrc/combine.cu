// Combine / unpermute: restore token order with the inverse map, apply the
// routing weights and sum each token's contributions ("MOE推理流程解析",
// section 三; section 二: T1's output is 0.7 * E1(T1) + 0.3 * E3(T1)).
//
//   out[t, :] = sum_{j<k} w[t, j] * y[inv_row[t*k + j], :]  (+ shared[t, :])
//
// fp32 accumulation in slot order j = 0..k-1, one rounding to the output
// dtype.  When the down projection was split along its reduction dimension,
// y holds S fp32 partial sums [S, R, d] that are added here (s = 0..S-1 in
// order) before the weight is applied.  Each thread owns 8 consecutive
// features of one token: 16-byte (bf16) or 2x16-byte (fp32) loads.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kMaxSplits = 8;  // the down GEMM uses at most 8 K splits

__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&a);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 a;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&a);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = a;
}

template <typename ActT, typename YT, bool SPLIT>
__global__ void __launch_bounds__(256) combine_kernel(int T, int k, int d, int R, int S,
                                                      const YT* __restrict__ y,
                                                      const int32_t* __restrict__ inv_row,
                                                      const float* __restrict__ w,
                                                      const ActT* __restrict__ shared,
                                                      ActT* __restrict__ out, int* status) {
  griddep_begin();
  const int groups = d / 8;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (long long)T * groups) return;
  const int t = (int)(gid / groups), c = (int)(gid % groups) * 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 4
  for (int j = 0; j < k; ++j) {
    const int r = inv_row[(size_t)t * k + j];
    if (r < 0 || r >= R) {
      set_device_status(status, MOE_ERR_DEVICE_BOUNDS);
      continue;
    }
    const float wj = w[(size_t)t * k + j];
    if (!SPLIT) {
      float part[8];
      load8(y + (size_t)r * d + c, part);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, part[i], acc[i]);
      continue;
    }
    // issue every partial's load before summing (split counts <= 8), so the
    // loads are in flight together; the sum is still in order s = 0..S-1
    float q[kMaxSplits][8];
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s)
      if (s < S) load8(y + ((size_t)s * R + r) * d + c, q[s]);
    float part[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) part[i] = q[0][i];
#pragma unroll
    for (int s = 1; s < kMaxSplits; ++s)
      if (s < S) {
#pragma unroll
        for (int i = 0; i < 8; ++i) part[i] += q[s][i];
      }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, part[i], acc[i]);
  }
  if (shared != nullptr) {
    float sv[8];
    load8(shared + (size_t)t * d + c, sv);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += sv[i];
  }
  store8(out + (size_t)t * d + c, acc);
}

}  // namespace

moe_status combine_launch(const CombineArgs& a, cudaStream_t s) {
  if (a.T == 0) return MOE_OK;
  if (a.y_partials > kMaxSplits) return MOE_ERR_UNSUPPORTED;
  if (a.d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  DeviceCtx ctx;
  MOE_TRY(device_ctx(&ctx));
  const long long work = (long long)a.T * (a.d / 8);
  const int blocks = (int)((work + 255) / 256);
  const int R = a.T * a.k;
  if (a.act_dtype == MOE_BF16) {
    const __nv_bfloat16* sh = static_cast<const __nv_bfloat16*>(a.shared);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    if (a.y_partials > 0)
      MOE_TRY_CUDA(launch_k(combine_kernel<__nv_bfloat16, float, true>, dim3(blocks), dim3(256), 0, s, 
          a.T, a.k, a.d, R, a.y_partials, static_cast<const float*>(a.y), a.inv_row, a.w, sh, out,
          ctx.status));
    else
      MOE_TRY_CUDA(launch_k(combine_kernel<__nv_bfloat16, __nv_bfloat16, false>, dim3(blocks), dim3(256), 0, s, 
          a.T, a.k, a.d, R, 1, static_cast<const __nv_bfloat16*>(a.y), a.inv_row, a.w, sh, out,
          ctx.status));
  } else if (a.act_dtype == MOE_F32) {
    if (a.y_partials > 1)
      MOE_TRY_CUDA(launch_k(combine_kernel<float, float, true>, dim3(blocks), dim3(256), 0, s,
          a.T, a.k, a.d, R, a.y_partials, static_cast<const float*>(a.y),
          a.inv_row, a.w, static_cast<const float*>(a.shared), static_cast<float*>(a.out),
          ctx.status));
    else
      MOE_TRY_CUDA(launch_k(combine_kernel<float, float, false>, dim3(blocks), dim3(256), 0, s,
          a.T, a.k, a.d, R, 1, static_cast<const float*>(a.y),
          a.inv_row, a.w, static_cast<const float*>(a.shared), static_cast<float*>(a.out),
          ctx.status));
  } else {
    return MOE_ERR_UNSUPPORTED;
  }
  MOE_TRY_CUDA(cudaGetLastError());
  return MOE_OK;
}

}  // namespace moe
