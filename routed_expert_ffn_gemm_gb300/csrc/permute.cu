// Dispatch on one GPU: group the T*k assignments by expert into contiguous
// row ranges, keep each row's source token id, record the inverse map, and
// move the token rows ("MOE推理流程解析", section 二: E1 receives T1, T2, T3
// -> a 3-row matrix, the source token id kept beside each row; section 三:
// the permutation writes token vectors in expert order and records an
// inverse map for the combine).
//
// Deterministic and bit-exact: a row's position inside its expert is the
// number of earlier assignments (in (t, j) order) to the same expert, found
// with warp match_any + popc and prefix sums over warps, chunks and experts;
// no result depends on the order of atomic operations.
//
//   small path  (R <= 2048): one block computes every map;
//   chunked path (any R):    count per 256-assignment chunk, one scan block,
//                            then per chunk: ranks and maps;
// then a grid-wide row gather moves x -> x_perm (one warp per row; the
// chunked blocks are too few to move rows at full bandwidth themselves).
// Row moves are 16-byte vector loads/stores, one warp per row.  When the
// experts run on f16 operands (FP8 weights) the row move also rounds the
// bf16 token vector to f16 (saturating to the largest finite f16).
#include <cuda_fp16.h>

#include "common.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kChunk = 256;       // assignments per chunk (chunked path)
constexpr int kSmallMaxR = 2048;  // largest R for the single-block path
constexpr int kSmallWarps = 16;

// 8 bf16 -> 8 f16 (round to nearest, saturate to +-65504).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
  uint4 r;
  uint32_t* o = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(b[i]);
    uint32_t h;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(f.y), "f"(f.x));
    o[i] = h;
  }
  return r;
}

__device__ __forceinline__ uint4 move16(uint4 v, int to_f16) { return to_f16 ? bf16x8_to_f16x8(v) : v; }

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Block-wide inclusive scan of one int per thread (blockDim.x <= 1024).
__device__ int block_inclusive_scan(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    int t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += n;
    }
    if (lane < nw) warp_tot[lane] = t;
  }
  __syncthreads();
  if (warp > 0) v += warp_tot[warp - 1];
  __syncthreads();
  return v;
}

// One warp walks assignments [a0, a1) in order; for each valid assignment it
// returns (through lrank) its rank among same-expert assignments of this walk
// and accumulates per-expert counts in cnt[E].
__device__ __forceinline__ void warp_walk(const int32_t* __restrict__ idx, int a0, int a1, int E,
                                          int* cnt, int* lrank, int lrank_base, int* status) {
  const int lane = threadIdx.x & 31;
  for (int s = a0; s < a1; s += 32) {
    const int a = s + lane;
    int e = a < a1 ? idx[a] : -1;
    if (a < a1 && (e < 0 || e >= E)) {
      set_device_status(status, MOE_ERR_DEVICE_BOUNDS);
      e = -1;
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) lrank[a - lrank_base] = cnt[e] + __popc(peers & lanemask_lt());
    __syncwarp();
    if (e >= 0 && (31 - __clz(peers)) == lane) cnt[e] += __popc(peers);
    __syncwarp();
  }
}

// ---------------------------------------------------------------- small path
// smem: wcnt[kSmallWarps][E], lrank[R], warp_tot[32], base[E], and with
// top-k selection rows[kSmallWarps][E] floats.
// With `logits` the block first selects each token's top-k (one warp per
// token, its logits row staged in shared memory) into idx_out / w_out, and
// the permutation then reads those indices: one launch instead of two at
// small batches.
__global__ void __launch_bounds__(1024) permute_small_kernel(
    int R, int k, int E, const int32_t* idx, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ perm_token,
    int32_t* __restrict__ inv_row, int* status, const float* __restrict__ logits,
    int32_t* idx_out, float* __restrict__ w_out, int32_t* __restrict__ zero, size_t zero_n) {
  griddep_begin();
  for (size_t i = threadIdx.x; i < zero_n; i += blockDim.x) zero[i] = 0;
  extern __shared__ int sm[];
  int* wcnt = sm;                        // [kSmallWarps][E]
  int* lrank = wcnt + kSmallWarps * E;   // [R]
  int* warp_tot = lrank + R;             // [32]
  int* base = warp_tot + 32;             // [E]
  const int warp = threadIdx.x >> 5;
  if (logits != nullptr) {
    float* rows = reinterpret_cast<float*>(base + E);  // [kSmallWarps][E]
    const int lane = threadIdx.x & 31, T = R / k;
    if (warp < kSmallWarps) {
      float* row = rows + warp * E;
      for (int t = warp; t < T; t += kSmallWarps) {
        for (int e = lane; e < E; e += 32) row[e] = logits[(size_t)t * E + e];
        __syncwarp();
        topk_row(row, E, k, idx_out + (size_t)t * k, w_out + (size_t)t * k);
        __syncwarp();
      }
    }
    __syncthreads();  // the indices written above are read below
    idx = idx_out;
  }
  for (int i = threadIdx.x; i < kSmallWarps * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const int seg = (R + kSmallWarps - 1) / kSmallWarps;
  if (warp < kSmallWarps) {
    const int a0 = min(R, warp * seg), a1 = min(R, a0 + seg);
    warp_walk(idx, a0, a1, E, wcnt + warp * E, lrank, 0, status);
  }
  __syncthreads();
  // per expert: exclusive prefix over warps, total count
  int tot = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kSmallWarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
    base[e] = run;
  }
  __syncthreads();
  // exclusive scan of the per-expert totals (E <= blockDim.x)
  tot = threadIdx.x < E ? base[threadIdx.x] : 0;
  const int incl = block_inclusive_scan(tot, warp_tot);
  if (threadIdx.x < E) {
    counts[threadIdx.x] = tot;
    offsets[threadIdx.x] = incl - tot;
    base[threadIdx.x] = incl - tot;
    if (threadIdx.x == E - 1) offsets[E] = incl;
  }
  __syncthreads();
  for (int a = threadIdx.x; a < R; a += blockDim.x) {
    const int e = idx[a];
    if (e < 0 || e >= E) continue;
    const int w = a / seg;
    const int row = base[e] + wcnt[w * E + e] + lrank[a];
    perm_token[row] = a / k;
    inv_row[a] = row;
  }
}

// x_perm[r] = x[perm_token[r]] for r < offsets[E]; one warp per row.
__global__ void __launch_bounds__(256) gather_rows_kernel(int R, int E, int vec_per_row,
                                                          const int32_t* __restrict__ offsets,
                                                          const int32_t* __restrict__ perm_token,
                                                          const uint4* __restrict__ x,
                                                          uint4* __restrict__ x_perm, int to_f16) {
  griddep_begin();
  const int lane = threadIdx.x & 31;
  const int nrows = min(R, offsets[E]);
  for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < nrows; r += gridDim.x * 8) {
    const size_t src = (size_t)perm_token[r] * vec_per_row, dst = (size_t)r * vec_per_row;
#pragma unroll 4
    for (int v = lane; v < vec_per_row; v += 32) x_perm[dst + v] = move16(x[src + v], to_f16);
  }
}

// n elements of bf16 -> f16, 8 per thread.
__global__ void __launch_bounds__(256) bf16_to_f16_kernel(const uint4* __restrict__ src,
                                                          uint4* __restrict__ dst, size_t nvec) {
  griddep_begin();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nvec; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = bf16x8_to_f16x8(src[i]);
}

// -------------------------------------------------------------- chunked path
__global__ void __launch_bounds__(256) permute_count_kernel(int R, int E,
                                                            const int32_t* __restrict__ idx,
                                                            int32_t* __restrict__ chunk_cnt,
                                                            int32_t* __restrict__ zero, size_t zero_n) {
  griddep_begin();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < zero_n; i += (size_t)gridDim.x * blockDim.x)
    zero[i] = 0;
  extern __shared__ int cnt[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int a = blockIdx.x * kChunk + threadIdx.x;
  if (a < R) {
    const int e = idx[a];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);  // a count: order-independent
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_cnt[(size_t)blockIdx.x * E + e] = cnt[e];
}

// chunk_cnt[c][e] -> offsets[e] + sum_{c'<c} chunk_cnt[c'][e] (in place).
// One block of 1024 threads: experts along the lanes (loads coalesced over
// experts), the chunks split into 32 slices over the warps; per-slice sums
// combine through shared memory.  kScanGroups groups of 32 experts share a
// round (their loads in flight together, two barriers per round).  A first
// pass finds the per-expert totals (-> counts, offsets), a second writes
// the running sums.
constexpr int kScanGroups = 4;
__global__ void __launch_bounds__(1024) permute_scan_kernel(int n_chunks, int E,
                                                            int32_t* __restrict__ chunk_cnt,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets) {
  griddep_begin();
  __shared__ int part[kScanGroups][32][33];
  __shared__ int base_e[1024];
  __shared__ int warp_tot[32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int per = (n_chunks + 31) / 32;
  const int c0 = min(n_chunks, w * per), c1 = min(n_chunks, c0 + per);
  // this warp's slice sum of expert g0 + 32 gi + lane, for every group gi of
  // the round, into part[gi][w][lane]
  auto slice_sums = [&](int g0) {
    int sum[kScanGroups];
#pragma unroll
    for (int gi = 0; gi < kScanGroups; ++gi) sum[gi] = 0;
    for (int c = c0; c < c1; ++c)
#pragma unroll
      for (int gi = 0; gi < kScanGroups; ++gi) {
        const int e = g0 + 32 * gi + lane;
        if (e < E) sum[gi] += chunk_cnt[(size_t)c * E + e];
      }
#pragma unroll
    for (int gi = 0; gi < kScanGroups; ++gi) part[gi][w][lane] = sum[gi];
  };
  for (int g0 = 0; g0 < E; g0 += 32 * kScanGroups) {
    slice_sums(g0);
    __syncthreads();
    if (w < kScanGroups) {
      const int e = g0 + 32 * w + lane;
      if (e < E) {
        int t = 0;
        for (int i = 0; i < 32; ++i) t += part[w][i][lane];
        base_e[e] = t;
      }
    }
    __syncthreads();
  }
  const int e = threadIdx.x;
  const int tot = e < E ? base_e[e] : 0;
  const int incl = block_inclusive_scan(tot, warp_tot);
  if (e < E) {
    counts[e] = tot;
    offsets[e] = incl - tot;
    if (e == E - 1) offsets[E] = incl;
    base_e[e] = incl - tot;
  }
  __syncthreads();
  for (int g0 = 0; g0 < E; g0 += 32 * kScanGroups) {
    slice_sums(g0);
    __syncthreads();
#pragma unroll
    for (int gi = 0; gi < kScanGroups; ++gi) {
      const int e2 = g0 + 32 * gi + lane;
      if (e2 < E) {
        int run = base_e[e2];
        for (int i = 0; i < w; ++i) run += part[gi][i][lane];
        for (int c = c0; c < c1; ++c) {
          const int v = chunk_cnt[(size_t)c * E + e2];
          chunk_cnt[(size_t)c * E + e2] = run;
          run += v;
        }
      }
    }
    __syncthreads();
  }
}

// smem: wcnt[8][E], lrank[kChunk], rows[kChunk]
__global__ void __launch_bounds__(256) permute_scatter_kernel(
    int R, int k, int E, int vec_per_row, const int32_t* __restrict__ idx,
    const int32_t* __restrict__ chunk_base, int32_t* __restrict__ perm_token,
    int32_t* __restrict__ inv_row, const uint4* __restrict__ x, uint4* __restrict__ x_perm,
    int* status, int to_f16) {
  griddep_begin();
  extern __shared__ int sm[];
  int* wcnt = sm;                 // [8][E]
  int* lrank = wcnt + 8 * E;      // [kChunk]
  int* rows = lrank + kChunk;     // [kChunk]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * kChunk;
  for (int i = threadIdx.x; i < 8 * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const int a0 = min(R, c0 + warp * 32), a1 = min(R, a0 + 32);
  warp_walk(idx, a0, a1, E, wcnt + warp * E, lrank, c0, status);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = chunk_base[(size_t)blockIdx.x * E + e];
    for (int w = 0; w < 8; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  const int a = c0 + threadIdx.x;
  int row = -1;
  if (a < R) {
    const int e = idx[a];
    if (e >= 0 && e < E) {
      row = wcnt[warp * E + e] + lrank[threadIdx.x];
      perm_token[row] = a / k;
      inv_row[a] = row;
    }
  }
  rows[threadIdx.x] = row;
  __syncthreads();
  if (x_perm != nullptr) {
    const int n = min(kChunk, R - c0);
    for (int i = warp; i < n; i += 8) {
      const int r = rows[i];
      if (r < 0) continue;
      const size_t src = (size_t)((c0 + i) / k) * vec_per_row, dst = (size_t)r * vec_per_row;
      for (int v = lane; v < vec_per_row; v += 32) x_perm[dst + v] = move16(x[src + v], to_f16);
    }
  }
}

size_t small_smem(int R, int E, bool topk) {
  return sizeof(int) * ((size_t)kSmallWarps * E + R + 32 + E) + (topk ? sizeof(float) * kSmallWarps * E : 0);
}

}  // namespace

moe_status bf16_to_f16_launch(const void* src, void* dst, size_t n, cudaStream_t s) {
  if (n == 0) return MOE_OK;
  if (n % 8 != 0) return MOE_ERR_UNSUPPORTED;
  const size_t nvec = n / 8;
  const int blocks = (int)((nvec + 255) / 256 < 4096 ? (nvec + 255) / 256 : 4096);
  MOE_TRY_CUDA(launch_k(bf16_to_f16_kernel, dim3(blocks), dim3(256), 0, s, static_cast<const uint4*>(src), static_cast<uint4*>(dst), nvec));
  MOE_TRY_CUDA(cudaGetLastError());
  return MOE_OK;
}

size_t permute_scratch_bytes(int T, int k, int E) {
  const size_t R = (size_t)T * k;
  if (R <= (size_t)kSmallMaxR) return 0;
  return ((R + kChunk - 1) / kChunk) * (size_t)E * sizeof(int32_t);
}

int permute_small_max() { return kSmallMaxR; }

int permute_launch_count(int T, int k, bool move_rows) {
  const long long R = (long long)T * k;
  if (R == 0) return 0;
  return (R <= kSmallMaxR ? 1 : 3) + (move_rows ? 1 : 0);
}

// x_perm[r] = x[perm_token[r]] over a grid-stride of warps.
moe_status gather_launch(const PermuteArgs& a, int R, int vec_per_row, cudaStream_t s) {
  if (a.x_perm == nullptr) return MOE_OK;
  const int blocks = min(4096, (R + 7) / 8);
  MOE_TRY_CUDA(launch_k(gather_rows_kernel, dim3(blocks), dim3(256), 0, s, R, a.E, vec_per_row,
                        a.offsets, a.perm_token, static_cast<const uint4*>(a.x),
                        static_cast<uint4*>(a.x_perm), a.to_f16));
  return MOE_OK;
}

moe_status permute_launch(const PermuteArgs& a, cudaStream_t s) {
  const int R = a.T * a.k;
  if (R == 0) {
    MOE_TRY_CUDA(cudaMemsetAsync(a.counts, 0, sizeof(int32_t) * a.E, s));
    MOE_TRY_CUDA(cudaMemsetAsync(a.offsets, 0, sizeof(int32_t) * (a.E + 1), s));
    return MOE_OK;
  }
  if (a.E > 1024) return MOE_ERR_UNSUPPORTED;
  const int vec_per_row = (a.d * a.act_bytes) / 16;
  const bool topk = a.topk_logits != nullptr;
  if (topk && (R > kSmallMaxR || a.idx_out == nullptr || a.w_out == nullptr)) return MOE_ERR_INVALID_ARG;
  if (R <= kSmallMaxR) {
    const size_t smem = small_smem(R, a.E, topk);
    MOE_TRY_CUDA(cudaFuncSetAttribute(permute_small_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    MOE_TRY_CUDA(launch_k(permute_small_kernel, dim3(1), dim3(1024), smem, s, R, a.k, a.E, a.idx, a.counts, a.offsets,
                          a.perm_token, a.inv_row, a.status, a.topk_logits, a.idx_out, a.w_out, a.zero,
                          a.zero != nullptr ? a.zero_n : 0));
    MOE_TRY_CUDA(cudaGetLastError());
    return gather_launch(a, R, vec_per_row, s);
  }
  if (a.chunk_scratch == nullptr) return MOE_ERR_WORKSPACE;
  const int n_chunks = (R + kChunk - 1) / kChunk;
  MOE_TRY_CUDA(launch_k(permute_count_kernel, dim3(n_chunks), dim3(256), sizeof(int) * a.E, s, R, a.E, a.idx,
                        a.chunk_scratch, a.zero, a.zero != nullptr ? a.zero_n : 0));
  MOE_TRY_CUDA(cudaGetLastError());
  MOE_TRY_CUDA(launch_k(permute_scan_kernel, dim3(1), dim3(1024), 0, s, n_chunks, a.E, a.chunk_scratch, a.counts, a.offsets));
  MOE_TRY_CUDA(cudaGetLastError());
  const size_t smem = sizeof(int) * (8 * (size_t)a.E + 2 * kChunk);
  MOE_TRY_CUDA(cudaFuncSetAttribute(permute_scatter_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  MOE_TRY_CUDA(launch_k(permute_scatter_kernel, dim3(n_chunks), dim3(256), smem, s, 
      R, a.k, a.E, vec_per_row, a.idx, a.chunk_scratch, a.perm_token, a.inv_row,
      static_cast<const uint4*>(a.x), static_cast<uint4*>(nullptr), a.status, a.to_f16));
  MOE_TRY_CUDA(cudaGetLastError());
  return gather_launch(a, R, vec_per_row, s);
}

}  // namespace moe
