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

// The selection order of logits as one unsigned key: a larger key ranks
// first.  The logit's bits mapped monotonically, -0 folded into +0 (which
// the order ties) and every NaN at 1, below every number (whose keys are
// at least 0x007fffff, that of -inf).  0 stands for "no candidate".  Equal
// keys go to the lower expert index.
__device__ __forceinline__ uint32_t selection_key(float v) {
  const float c = __fadd_rn(v, 0.0f);  // -0 -> +0
  const uint32_t b = __float_as_uint(c);
  return c != c ? 1u : ((b & 0x80000000u) ? ~b : (b | 0x80000000u));
}

// One warp, lane j < k holding the logit and expert of slot j (slots in
// selection order): weights exp(l_j - l_0) / sum over the slots, written
// with the indices.
__device__ __forceinline__ void topk_weights(float my_v, int my_e, int k, int32_t* idx_out, float* w_out) {
  const int lane = threadIdx.x & 31;
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

// One warp: top-k of one token's logits row (shared or global memory).
// Round j: each lane's best untaken (key, index), then one warp max of the
// keys and one warp min of the indices holding it (redux.sync each); the
// winner's lane marks it taken.
__device__ inline void topk_row(const float* row, int E, int k, int32_t* idx_out, float* w_out) {
  const int lane = threadIdx.x & 31;
  const int per_lane = (E + 31) / 32;  // <= 32
  uint32_t taken = 0;                  // bit i: expert lane + 32*i already chosen
  float my_v = 0.f;
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t key = 0u, e_best = 0xffffffffu;
    for (int i = 0; i < per_lane; ++i) {  // ascending index: the strict > keeps the lower one
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u)) {
        const uint32_t ke = selection_key(row[e]);
        if (ke > key) {
          key = ke;
          e_best = (uint32_t)e;
        }
      }
    }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);  // E >= k: an untaken expert remains
    const int be = (int)__reduce_min_sync(0xffffffffu, key == kmax ? e_best : 0xffffffffu);
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) {
      my_e = be;
      my_v = row[be];
    }
  }
  topk_weights(my_v, my_e, k, idx_out, w_out);
}

}  // namespace moe
