// Per-row E4M3 quantisation of activation rows for the FP8-activation mode
// of the routed experts ("MOE推理流程解析", section 三: the activations may
// be quantised before dispatch, so the permuted rows carry fewer bytes;
// "MoE 推理部署", section 专家量化: FP8 inference): the token rows before
// the gate/up GEMM, the rows of h before the down GEMM.
//
// Row t of x [rows, d] (bf16, or f16: the rows of h) becomes
//   s_t     = max_i |x[t,i]| / 448     (1 for an all-zero row)
//   q[t,i]  = E4M3(x[t,i] / s_t)       round to nearest, ties to even,
//                                      magnitudes past 448 saturate to 448
// with both divisions correctly rounded in fp32, so that the codes are a
// function of the stored inputs alone.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kQThreads = 128;

// The two 16-bit values of a word as fp32 (exact): bf16, or f16.
template <bool F16>
__device__ __forceinline__ float lo16(uint32_t w) {
  if constexpr (F16) return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
  return __uint_as_float(w << 16);
}
template <bool F16>
__device__ __forceinline__ float hi16(uint32_t w) {
  if constexpr (F16) return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
  return __uint_as_float(w & 0xffff0000u);
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// One CTA per row (grid-stride over rows); each thread takes 8 elements
// (16 bytes) at a time.  Pass 1 finds the row's absolute maximum, pass 2
// re-reads the row (L1/L2-resident: at most a few tens of KB) and writes the
// codes, 8 bytes per thread.
template <bool F16>
__global__ void __launch_bounds__(kQThreads) quantize_rows_e4m3_kernel(const uint4* __restrict__ x, int rows,
                                                                       int vpr, uint2* __restrict__ codes,
                                                                       float* __restrict__ scales) {
  griddep_begin();
  __shared__ float red[kQThreads / 32];
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint4* xr = x + (size_t)r * vpr;
    float m = 0.f;
    for (int v = threadIdx.x; v < vpr; v += kQThreads) {
      const uint4 q = xr[v];
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(lo16<F16>(w[i])), fabsf(hi16<F16>(w[i]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int i = 1; i < kQThreads / 32; ++i) amax = fmaxf(amax, red[i]);
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    if (threadIdx.x == 0) scales[r] = s;
    uint2* cr = codes + (size_t)r * vpr;
    for (int v = threadIdx.x; v < vpr; v += kQThreads) {
      const uint4 q = xr[v];
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
      uint32_t c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) c[i] = e4m3x2(__fdiv_rn(lo16<F16>(w[i]), s), __fdiv_rn(hi16<F16>(w[i]), s));
      cr[v] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    }
    __syncthreads();  // red[] is rewritten by the next row
  }
}

// Two-term E4M3 encoding of bf16 rows: the bf16 values themselves for
// every element within 2^9 of its row's largest magnitude, and within
// s * 2^-10 below that:
//   s_t      = 2^p, p the integer with max_i |x[t,i]| / 2^p in (224, 448]
//              (1 for an all-zero row)
//   hi[t,i]  = E4M3(x[t,i] / s_t)                        round to nearest even
//   lo[t,i]  = E4M3(x[t,i] / s_t - hi[t,i])              round to nearest even
//   x[t,i]   = s_t * (hi[t,i] + lo[t,i])
// A bf16 value a = x / s has 8 significant bits: hi keeps the top four
// (rounded) and the remainder a - hi, at most half of hi's step, is a
// signed 3-bit multiple of a's own last bit, 2^(e-7) for a in [2^e,
// 2^(e+1)); E4M3 holds that exactly while 2^(e-7) >= 2^-9, its smallest
// step, i.e. for a >= 2^-2 (|x| >= s / 4 >= max |x| / 896).  Dividing by a
// power of two is exact, and so is the subtraction in fp32.  Codes
// [2, rows, d]: the hi codes of every row, then the lo codes (plane p, row
// t at row p * rows + t of a [2 * rows, d] byte matrix).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
  return __half2float(__half(h));
}

// With dst_rows (scatter form): row t's codes and scale go to rows
// dst_rows[t*k + j], j < k, of planes of R rows (an out-of-range row is
// recorded as MOE_ERR_DEVICE_BOUNDS and skipped); else to row t of planes
// of `rows` rows.
template <bool F16>
__global__ void __launch_bounds__(kQThreads) split_rows_e4m3x2_kernel(const uint4* __restrict__ x, int rows,
                                                                      int vpr, uint2* __restrict__ codes,
                                                                      float* __restrict__ scales,
                                                                      const int32_t* __restrict__ dst_rows, int k,
                                                                      int R, int* status) {
  griddep_begin();
  __shared__ float red[kQThreads / 32];
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint4* xr = x + (size_t)r * vpr;
    float m = 0.f;
    for (int v = threadIdx.x; v < vpr; v += kQThreads) {
      const uint4 q = xr[v];
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(lo16<F16>(w[i])), fabsf(hi16<F16>(w[i]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int i = 1; i < kQThreads / 32; ++i) amax = fmaxf(amax, red[i]);
    // amax = f * 2^e with f in [0.5, 1): p = e - 9 puts amax / 2^p in
    // [256, 448] when f <= 0.875, else p = e - 8 puts it in (224, 256)
    int e = 0;
    const float f = frexpf(amax, &e);
    const int p = amax > 0.f ? (f <= 0.875f ? e - 9 : e - 8) : 0;
    // x / 2^p as two exact power-of-two factors (each within fp32's range)
    const float inv_a = ldexpf(1.f, -(p / 2)), inv_b = ldexpf(1.f, -(p - p / 2));
    // destination rows of this row's codes (one, or its k permuted rows)
    const int nd = dst_rows != nullptr ? k : 1;
    const int plane = dst_rows != nullptr ? R : rows;
    if (threadIdx.x < nd) {
      const int dr = dst_rows != nullptr ? dst_rows[(size_t)r * k + threadIdx.x] : r;
      if (dr >= 0 && dr < plane)
        scales[dr] = ldexpf(1.f, p);
      else
        set_device_status(status, MOE_ERR_DEVICE_BOUNDS);
    }
    for (int v = threadIdx.x; v < vpr; v += kQThreads) {
      const uint4 q = xr[v];
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
      uint32_t ch[4], cl[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = lo16<F16>(w[i]) * inv_a * inv_b, b = hi16<F16>(w[i]) * inv_a * inv_b;
        ch[i] = e4m3x2(a, b);
        const float ra = a - e4m3_value(ch[i] & 0xffu), rb = b - e4m3_value(ch[i] >> 8);
        cl[i] = e4m3x2(ra, rb);
      }
      const uint2 hv = make_uint2(ch[0] | (ch[1] << 16), ch[2] | (ch[3] << 16));
      const uint2 lv = make_uint2(cl[0] | (cl[1] << 16), cl[2] | (cl[3] << 16));
      for (int j = 0; j < nd; ++j) {
        const int dr = dst_rows != nullptr ? __ldg(dst_rows + (size_t)r * k + j) : r;
        if (dr < 0 || dr >= plane) continue;
        codes[(size_t)dr * vpr + v] = hv;
        codes[(size_t)(plane + dr) * vpr + v] = lv;
      }
    }
    __syncthreads();  // red[] is rewritten by the next row
  }
}

// The same split with the row held in registers (NV 16-byte vectors per
// thread, rows of up to NV * 128 * 8 elements): no second read of the row,
// and each CTA loads its next row while it reduces and writes the current
// one, so twice the rows are in flight per SM.  Same arithmetic, same codes.
template <bool F16, int NV>
__global__ void __launch_bounds__(kQThreads) split_rows_e4m3x2_regs_kernel(const uint4* __restrict__ x, int rows,
                                                                           int vpr, uint2* __restrict__ codes,
                                                                           float* __restrict__ scales,
                                                                           const int32_t* __restrict__ dst_rows,
                                                                           int k, int R, int* status) {
  griddep_begin();
  __shared__ float red[2][kQThreads / 32];  // by row parity: no barrier needed after a row
  auto load_row = [&](int r, uint4 (&buf)[NV]) {
    const uint4* xr = x + (size_t)r * vpr;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int v = threadIdx.x + i * kQThreads;
      buf[i] = v < vpr ? xr[v] : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  uint4 cur[NV], nxt[NV];
  int r = blockIdx.x;
  if (r < rows) load_row(r, cur);
  for (int it = 0; r < rows; r += gridDim.x, ++it) {
    if (r + (int)gridDim.x < rows) load_row(r + gridDim.x, nxt);
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const uint32_t w[4] = {cur[i].x, cur[i].y, cur[i].z, cur[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(lo16<F16>(w[j])), fabsf(hi16<F16>(w[j]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float* rd = red[it & 1];
    if ((threadIdx.x & 31) == 0) rd[threadIdx.x >> 5] = m;
    __syncthreads();
    float amax = rd[0];
#pragma unroll
    for (int i = 1; i < kQThreads / 32; ++i) amax = fmaxf(amax, rd[i]);
    int e = 0;
    const float f = frexpf(amax, &e);
    const int p = amax > 0.f ? (f <= 0.875f ? e - 9 : e - 8) : 0;
    const float inv_a = ldexpf(1.f, -(p / 2)), inv_b = ldexpf(1.f, -(p - p / 2));
    const int nd = dst_rows != nullptr ? k : 1;
    const int plane = dst_rows != nullptr ? R : rows;
    if (threadIdx.x < nd) {
      const int dr = dst_rows != nullptr ? dst_rows[(size_t)r * k + threadIdx.x] : r;
      if (dr >= 0 && dr < plane)
        scales[dr] = ldexpf(1.f, p);
      else
        set_device_status(status, MOE_ERR_DEVICE_BOUNDS);
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int v = threadIdx.x + i * kQThreads;
      if (v >= vpr) break;
      const uint32_t w[4] = {cur[i].x, cur[i].y, cur[i].z, cur[i].w};
      uint32_t ch[4], cl[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a = lo16<F16>(w[j]) * inv_a * inv_b, b = hi16<F16>(w[j]) * inv_a * inv_b;
        ch[j] = e4m3x2(a, b);
        const float ra = a - e4m3_value(ch[j] & 0xffu), rb = b - e4m3_value(ch[j] >> 8);
        cl[j] = e4m3x2(ra, rb);
      }
      const uint2 hv = make_uint2(ch[0] | (ch[1] << 16), ch[2] | (ch[3] << 16));
      const uint2 lv = make_uint2(cl[0] | (cl[1] << 16), cl[2] | (cl[3] << 16));
      for (int j = 0; j < nd; ++j) {
        const int dr = dst_rows != nullptr ? __ldg(dst_rows + (size_t)r * k + j) : r;
        if (dr < 0 || dr >= plane) continue;
        codes[(size_t)dr * vpr + v] = hv;
        codes[(size_t)(plane + dr) * vpr + v] = lv;
      }
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) cur[i] = nxt[i];
  }
}

// One of the split kernels for rows of vpr 16-byte vectors: the register
// form when the row fits 4 vectors per thread, else the two-pass form (with
// 8 vectors per thread the register form holds 121 registers, 4 CTAs per
// SM, and fewer rows in flight than the two-pass form's 16 CTAs).
template <bool F16>
moe_status launch_split(int blocks, cudaStream_t s, const uint4* x, int rows, int vpr, uint2* codes,
                        float* scales, const int32_t* dst_rows, int k, int R, int* status) {
  const int nv = (vpr + kQThreads - 1) / kQThreads;
  if (nv <= 1)
    MOE_TRY_CUDA(launch_k(split_rows_e4m3x2_regs_kernel<F16, 1>, dim3(blocks), dim3(kQThreads), 0, s, x, rows, vpr,
                          codes, scales, dst_rows, k, R, status));
  else if (nv <= 2)
    MOE_TRY_CUDA(launch_k(split_rows_e4m3x2_regs_kernel<F16, 2>, dim3(blocks), dim3(kQThreads), 0, s, x, rows, vpr,
                          codes, scales, dst_rows, k, R, status));
  else if (nv <= 4)
    MOE_TRY_CUDA(launch_k(split_rows_e4m3x2_regs_kernel<F16, 4>, dim3(blocks), dim3(kQThreads), 0, s, x, rows, vpr,
                          codes, scales, dst_rows, k, R, status));
  else
    MOE_TRY_CUDA(launch_k(split_rows_e4m3x2_kernel<F16>, dim3(blocks), dim3(kQThreads), 0, s, x, rows, vpr, codes,
                          scales, dst_rows, k, R, status));
  MOE_TRY_CUDA(cudaGetLastError());
  return MOE_OK;
}

}  // namespace

moe_status split_rows_e4m3x2_launch(const void* x, int rows, int d, void* codes, float* scales, int num_sms,
                                    cudaStream_t s, bool f16_in) {
  if (rows == 0) return MOE_OK;
  if (rows < 0 || d <= 0 || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  const int blocks = rows < 16 * num_sms ? rows : 16 * num_sms;
  const uint4* xv = static_cast<const uint4*>(x);
  uint2* cv = static_cast<uint2*>(codes);
  return f16_in ? launch_split<true>(blocks, s, xv, rows, d / 8, cv, scales, nullptr, 1, rows, nullptr)
                : launch_split<false>(blocks, s, xv, rows, d / 8, cv, scales, nullptr, 1, rows, nullptr);
}

moe_status split_rows_e4m3x2_scatter_launch(const void* x, int T, int d, int k, const int32_t* dst_rows, int R,
                                            void* codes, float* scales, int* status, int num_sms,
                                            cudaStream_t s) {
  if (T == 0) return MOE_OK;
  if (T < 0 || d <= 0 || d % 8 != 0 || k < 1 || k > kQThreads || dst_rows == nullptr) return MOE_ERR_UNSUPPORTED;
  const int blocks = T < 16 * num_sms ? T : 16 * num_sms;
  return launch_split<false>(blocks, s, static_cast<const uint4*>(x), T, d / 8, static_cast<uint2*>(codes), scales,
                             dst_rows, k, R, status);
}

moe_status quantize_rows_e4m3_launch(const void* x, int rows, int d, void* codes, float* scales,
                                     int num_sms, cudaStream_t s, bool f16_in) {
  if (rows == 0) return MOE_OK;
  if (rows < 0 || d <= 0 || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  const int blocks = rows < 16 * num_sms ? rows : 16 * num_sms;
  if (f16_in)
    MOE_TRY_CUDA(launch_k(quantize_rows_e4m3_kernel<true>, dim3(blocks), dim3(kQThreads), 0, s,
                          static_cast<const uint4*>(x), rows, d / 8, static_cast<uint2*>(codes), scales));
  else
    MOE_TRY_CUDA(launch_k(quantize_rows_e4m3_kernel<false>, dim3(blocks), dim3(kQThreads), 0, s,
                          static_cast<const uint4*>(x), rows, d / 8, static_cast<uint2*>(codes), scales));
  MOE_TRY_CUDA(cudaGetLastError());
  return MOE_OK;
}

}  // namespace moe
