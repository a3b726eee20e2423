// fp32 grouped SwiGLU experts on the CUDA cores (fp32 storage, fp32 FMA,
// no TF32), for layers stored in fp32 ("MOE推理流程解析", section 三: each
// expert applies its activation and output projection to its own rows).
//
//   h[r, :] = SiLU(x_perm[r, :] W_g[e]^T) * (x_perm[r, :] W_u[e]^T)
//   y[r, :] = h[r, :] W_d[e]^T          for r in [offsets[e], offsets[e+1])
//
// One block per row (grid-stride), the row staged in shared memory, one warp
// per output feature with coalesced loads of the weight row and a shuffle
// reduction.
#include "common.cuh"

namespace moe {
namespace {

// The expert whose row range holds r, or -1 if none does.
__device__ __forceinline__ int expert_of_row(const int32_t* __restrict__ offsets, int E, int r) {
  if (r < offsets[0] || r >= offsets[E]) return -1;
  int lo = 0, hi = E - 1;  // largest e with offsets[e] <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (offsets[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(256) simt_gateup_kernel(int R, int d, int ffn, int E,
                                                          const float* __restrict__ x,
                                                          const int32_t* __restrict__ offsets,
                                                          const float* __restrict__ wg,
                                                          const float* __restrict__ wu,
                                                          float* __restrict__ h) {
  griddep_begin();
  extern __shared__ float xs[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = blockIdx.x; r < R; r += gridDim.x) {
    const int e = expert_of_row(offsets, E, r);
    if (e < 0) continue;  // uniform across the block
    __syncthreads();
    for (int i = threadIdx.x; i < d; i += blockDim.x) xs[i] = x[(size_t)r * d + i];
    __syncthreads();
    for (int c = warp; c < ffn; c += 8) {
      const float* g = wg + ((size_t)e * ffn + c) * d;
      const float* u = wu + ((size_t)e * ffn + c) * d;
      float sg = 0.f, su = 0.f;
      for (int i = lane; i < d; i += 32) {
        sg = fmaf(xs[i], g[i], sg);
        su = fmaf(xs[i], u[i], su);
      }
      sg = warp_sum(sg);
      su = warp_sum(su);
      if (lane == 0) h[(size_t)r * ffn + c] = sg / (1.f + expf(-sg)) * su;
    }
  }
}

__global__ void __launch_bounds__(256) simt_down_kernel(int R, int d, int ffn, int E,
                                                        const float* __restrict__ h,
                                                        const int32_t* __restrict__ offsets,
                                                        const float* __restrict__ wd,
                                                        float* __restrict__ y) {
  griddep_begin();
  extern __shared__ float hs[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = blockIdx.x; r < R; r += gridDim.x) {
    const int e = expert_of_row(offsets, E, r);
    if (e < 0) continue;
    __syncthreads();
    for (int i = threadIdx.x; i < ffn; i += blockDim.x) hs[i] = h[(size_t)r * ffn + i];
    __syncthreads();
    for (int c = warp; c < d; c += 8) {
      const float* wrow = wd + ((size_t)e * d + c) * ffn;
      float s = 0.f;
      for (int i = lane; i < ffn; i += 32) s = fmaf(hs[i], wrow[i], s);
      s = warp_sum(s);
      if (lane == 0) y[(size_t)r * d + c] = s;
    }
  }
}

}  // namespace

moe_status simt_grouped_launch(const SimtGroupedArgs& a, cudaStream_t s, cudaEvent_t mid) {
  if (a.R == 0) return MOE_OK;
  const size_t smem_g = sizeof(float) * a.d, smem_d = sizeof(float) * a.ffn;
  if (smem_g > 200 * 1024 || smem_d > 200 * 1024) return MOE_ERR_UNSUPPORTED;
  MOE_TRY_CUDA(cudaFuncSetAttribute(simt_gateup_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_g));
  MOE_TRY_CUDA(cudaFuncSetAttribute(simt_down_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_d));
  const int blocks = a.R < 65535 ? a.R : 65535;
  MOE_TRY_CUDA(launch_k(simt_gateup_kernel, dim3(blocks), dim3(256), smem_g, s, a.R, a.d, a.ffn, a.E, a.x_perm, a.offsets,
                                                 a.w_gate, a.w_up, a.h));
  MOE_TRY_CUDA(cudaGetLastError());
  if (mid != nullptr) MOE_TRY_CUDA(record_event(mid, s));
  MOE_TRY_CUDA(launch_k(simt_down_kernel, dim3(blocks), dim3(256), smem_d, s, a.R, a.d, a.ffn, a.E, a.h, a.offsets, a.w_down,
                                               a.y));
  MOE_TRY_CUDA(cudaGetLastError());
  return MOE_OK;
}

}  // namespace moe
