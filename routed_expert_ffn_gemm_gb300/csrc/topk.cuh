// Per-token top-k selection over a row of router logits, shared by the
// router and the fused small-batch permutation.
//
// Selection: k rounds of a warp arg-max over the E logits (larger logit
// first, ties to the lower expert index; NaN logits last).  Weights:
// exp(l_j - l_max) / sum over the kept set, which equals p_j / sum_{kept} p
// with p = softmax over all E (the full-softmax denominator cancels), as
// "MOE推理流程解析" section 三 (top-k keeps indices and weights) and
// section 九 (the kept weights are re-normalised) define.  Slots are in
// selection order, i.e. descending weight.
#pragma once

#include <math.h>
#include <stdint.h>

namespace moe {

// (v1, e1) ranks before (v2, e2): larger logit, ties to the lower index.
__device__ __forceinline__ bool ranks_before(float v1, int e1, float v2, int e2) {
  return v1 > v2 || (v1 == v2 && e1 < e2);
}

// One warp: top-k of one token's logits row (shared or global memory).
__device__ inline void topk_row(const float* row, int E, int k, int32_t* idx_out, float* w_out) {
  const int lane = threadIdx.x & 31;
  const int per_lane = (E + 31) / 32;  // <= 32
  uint32_t taken = 0;                  // bit i: expert lane + 32*i already chosen
  float my_v = 0.f;
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = E;  // E = no candidate
    for (int i = 0; i < per_lane; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u)) {
        const float v = row[e];
        if (ranks_before(v, e, bv, be)) { bv = v; be = e; }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ranks_before(ov, oe, bv, be)) { bv = ov; be = oe; }
    }
    if (be >= E) {  // only NaN logits remain: take the lowest unchosen expert
      int le = E;
      for (int i = 0; i < per_lane; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u)) { le = e; break; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) le = min(le, __shfl_xor_sync(0xffffffffu, le, o));
      be = le;
      bv = row[be];
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) { my_v = bv; my_e = be; }
  }
  const float vmax = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < k ? expf(my_v - vmax) : 0.f;
  float s = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane < k) {
    idx_out[lane] = my_e;
    w_out[lane] = ex / s;
  }
}

}  // namespace moe
