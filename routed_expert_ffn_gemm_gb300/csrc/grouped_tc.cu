// Grouped SwiGLU expert GEMMs on the 5th-generation tensor cores (tcgen05,
// TMEM accumulators, TMA-fed shared-memory pipeline) for sm_103a.
//
// "MOE推理流程解析", section 三: a grouped GEMM runs several expert matrices
// with different row counts in one launch, grouping changes the number of
// launches but not the content; each expert then applies its activation and
// output projection.  Section 二: prefill gives experts many rows, decode
// one or two (the degenerate, batched-GEMV case).
//
// Orientation ("swap-AB"): the MMA's M = 128 side is a tile of 128 output
// channels of one expert's weight matrix (operand A, K-major), and its N side
// is the expert's assignment rows (operand B, K-major, N = 16..BN in steps of
// 16).  Weights are therefore always full tiles, and a group with n rows costs
// ceil(n/16)*16 MMA columns: the decode regime (1-2 rows per expert) and the
// prefill regime (hundreds of rows) run the same kernel.
//
// Work unit = (expert g, tile of BN rows, 128-channel tile mt, K split ks).
// A persistent grid (one CTA per SM) strides over the units; the per-expert
// tile counts are derived on the device from the offsets (no host sync).
// CTA roles (192 threads):
//   warp 0 lane 0   TMA producer: weight tile(s) [128 x 64] + ceil(n/16)
//                   row boxes [16 x 64] per stage, 128-byte swizzle
//   warp 1 lane 0   MMA issuer: tcgen05.mma kind::f16, fp32 accumulate;
//                   warp 1 also allocates / frees 512 TMEM columns
//   warps 2..5      epilogue: tcgen05.ld from TMEM, SiLU(g)*u (gate/up) or
//                   the projection (down), 64/128-byte coalesced stores
// Accumulators are double-buffered in TMEM (buffer b at column 256*b; gate at
// +0, up at +128) so the epilogue of one unit overlaps the next unit's loads
// and MMAs.  Every wait is bounded: on expiry the kernel records
// MOE_ERR_DEVICE_TIMEOUT, lets issued copies land, frees TMEM and returns.
#include <string.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;          // output channels per tile (MMA M)
constexpr int kBK = 64;           // reduction elements per stage (128 bytes of bf16)
constexpr int kBoxN = 16;         // rows per B box
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxGroups = 1024;
constexpr int kSmemLimit = 232448;  // opt-in maximum dynamic shared memory per block

enum { kGateUp = 0, kDown = 1 };

struct TcParams {
  int G;
  const int32_t* offsets;  // [G+1]
  int R;                   // rows of B and of the outputs
  int M;                   // output channels per group
  int K;                   // reduction length
  int splits;              // K splits (down GEMM)
  void* out;               // gate/up: h bf16 [R, M]; down: bf16 [R, M] or fp32 [splits, R, M]
  int out_f32;
  int* status;
  long long timeout_ns;
  int selftest;            // 1: issue no copies/MMAs, wait on a barrier nothing arrives at
};

template <int MODE, int BN>
struct Cfg {
  static constexpr int NA = MODE == kGateUp ? 2 : 1;           // weight operands per stage
  static constexpr int A_BYTES = kBM * kBK * 2;                // 16 KB
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int STAGE_BYTES = NA * A_BYTES + B_BYTES;   // multiple of 1024
  static constexpr int TAIL_BYTES = 8 * 24 + 16 + 4 * 2 * (kMaxGroups + 8);
  static constexpr int STAGES_FIT = (kSmemLimit - 1024 - TAIL_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 10 ? 10 : STAGES_FIT;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  // barriers: full[S], empty[S], acc_full[2], acc_empty[2], drain
  static constexpr int NBARS = 2 * STAGES + 5;
  static constexpr int SLOT_OFF = BAR_OFF + 8 * NBARS;         // TMEM base address
  static constexpr int ABORT_OFF = SLOT_OFF + 8;
  static constexpr int OFFS_OFF = ABORT_OFF + 8;               // int offs[G+1]
  static constexpr int PREFIX_OFF = OFFS_OFF + 4 * (kMaxGroups + 4);
  static constexpr int SMEM_BYTES = PREFIX_OFF + 4 * (kMaxGroups + 4) + 1024;
  static_assert(STAGES >= 2, "pipeline too shallow");
  static_assert(SMEM_BYTES <= kSmemLimit, "shared memory budget");
  static_assert(BN % kBoxN == 0 && BN <= (MODE == kGateUp ? 128 : 256), "tile rows");
};

struct Unit {
  int g, row0, n_valid, mt, ks;
};

__device__ __forceinline__ Unit decode_unit(int u, const int* offs, const int* prefix, int G,
                                            int MT, int S, int BN) {
  Unit x;
  x.ks = u % S;
  const int t = u / S;
  x.mt = t % MT;
  const int tile = t / MT;
  int lo = 0, hi = G - 1;  // largest g with prefix[g] <= tile: that group owns the tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  x.g = lo;
  const int n0 = (tile - prefix[lo]) * BN;
  const int cnt = max(0, offs[lo + 1] - offs[lo]);
  x.row0 = offs[lo] + n0;
  x.n_valid = min(BN, cnt - n0);
  return x;
}

__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <int MODE, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    tc_grouped_kernel(const TcParams p, const __grid_constant__ CUtensorMap tmA0,
                      const __grid_constant__ CUtensorMap tmA1,
                      const __grid_constant__ CUtensorMap tmB) {
  using C = Cfg<MODE, BN>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = ptx::smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_s + pad;
  const uint32_t bars = sbase + C::BAR_OFF;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (2 * STAGES + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::SLOT_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::ABORT_OFF);
  int* offs = reinterpret_cast<int*>(smem + C::OFFS_OFF);
  int* prefix = reinterpret_cast<int*>(smem + C::PREFIX_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t deadline = ptx::globaltimer_ns() + (uint64_t)p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(accf_bar(b), 1);
      ptx::mbar_init(acce_bar(b), 4);  // one arrival per epilogue warp
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0 && !p.selftest) {
    ptx::prefetch_tmap(&tmA0);
    if (MODE == kGateUp) ptx::prefetch_tmap(&tmA1);
    ptx::prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }

  // Group row ranges (clamped into [0, R]) and the exclusive prefix of
  // per-group tile counts ceil(rows / BN).
  const int G = p.selftest ? 1 : p.G;
  for (int g = threadIdx.x; g <= G; g += kThreads) {
    int o = p.selftest ? 0 : p.offsets[g];
    if (o < 0 || o > p.R) {
      set_device_status(p.status, MOE_ERR_DEVICE_BOUNDS);
      o = o < 0 ? 0 : p.R;
    }
    offs[g] = o;
  }
  __syncthreads();
  {
    const int per = (G + kThreads - 1) / kThreads;
    const int g0 = min(G, threadIdx.x * per), g1 = min(G, g0 + per);
    int local = 0;
    for (int g = g0; g < g1; ++g) local += (max(0, offs[g + 1] - offs[g]) + BN - 1) / BN;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    __shared__ int warp_sum[kThreads / 32];
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += warp_sum[w];
    int run = before + incl - local;
    for (int g = g0; g < g1; ++g) {
      prefix[g] = run;
      run += (max(0, offs[g + 1] - offs[g]) + BN - 1) / BN;
    }
    if (threadIdx.x == kThreads - 1) prefix[G] = before + incl;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int MT = p.M / kBM;
  const int S = p.splits;
  const int total_units = p.selftest ? 1 : prefix[G] * MT * S;
  const int kblocks = (p.K + kBK - 1) / kBK;
  const int kb_per_split = (kblocks + S - 1) / S;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !p.selftest) {
      const uint64_t pol_w = ptx::policy_evict_first();
      const uint64_t pol_x = ptx::policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int armed[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) armed[s] = -1;
      bool ok = true;
      for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
        const Unit x = decode_unit(u, offs, prefix, G, MT, S, BN);
        const int kb0 = x.ks * kb_per_split, kb1 = min(kblocks, kb0 + kb_per_split);
        const int nbox = (x.n_valid + kBoxN - 1) / kBoxN;
        const uint32_t bytes = C::NA * C::A_BYTES + nbox * kBoxN * kBK * 2;
        const int arow = x.g * p.M + x.mt * kBM;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait_bounded(empty_bar(stage), phase ^ 1u, deadline, abort_flag)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(full_bar(stage), bytes);
          armed[stage] = (int)phase;
          const uint32_t sa = sbase + stage * C::STAGE_BYTES;
          ptx::tma_load_2d(sa, &tmA0, full_bar(stage), kb * kBK, arow, pol_w);
          if (MODE == kGateUp) ptx::tma_load_2d(sa + C::A_BYTES, &tmA1, full_bar(stage), kb * kBK, arow, pol_w);
          const uint32_t sb = sa + C::NA * C::A_BYTES;
          for (int i = 0; i < nbox; ++i)
            ptx::tma_load_2d(sb + i * kBoxN * kBK * 2, &tmB, full_bar(stage), kb * kBK,
                             x.row0 + i * kBoxN, pol_x);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        set_device_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
        // let every issued copy land before shared memory is released
        const uint64_t grace = ptx::globaltimer_ns() + 100000000ull;
        for (int s = 0; s < STAGES; ++s) {
          if (armed[s] < 0) continue;
          while (!ptx::mbar_try_wait(full_bar(s), (uint32_t)armed[s]) && ptx::globaltimer_ns() < grace) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      bool issued = false;
      if (p.selftest) {
        // nothing ever arrives on full_bar(0): the wait must expire
        ok = ptx::mbar_wait_bounded(full_bar(0), 0u, deadline, abort_flag);
      } else {
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x, ++it) {
          const Unit x = decode_unit(u, offs, prefix, G, MT, S, BN);
          const int kb0 = x.ks * kb_per_split, kb1 = min(kblocks, kb0 + kb_per_split);
          const int buf = it & 1;
          const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
          if (!ptx::mbar_wait_bounded(acce_bar(buf), acc_phase ^ 1u, deadline, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const int n_mma = ((x.n_valid + 15) / 16) * 16;
          const uint32_t idesc = ptx::idesc_bf16_f32(kBM, n_mma);
          const uint32_t d0 = tmem_base + 256u * buf;
          const uint32_t d1 = d0 + 128u;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!ptx::mbar_wait_bounded(full_bar(stage), phase, deadline, abort_flag)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t sa = sbase + stage * C::STAGE_BYTES;
            const uint64_t da0 = ptx::sdesc_k_sw128(sa);
            const uint64_t da1 = ptx::sdesc_k_sw128(sa + C::A_BYTES);
            const uint64_t db = ptx::sdesc_k_sw128(sa + C::NA * C::A_BYTES);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
              ptx::mma_f16(d0, da0 + 2 * kk, db + 2 * kk, idesc, acc);
              if (MODE == kGateUp) ptx::mma_f16(d1, da1 + 2 * kk, db + 2 * kk, idesc, acc);
            }
            issued = true;
            ptx::mma_commit(empty_bar(stage));
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) ptx::mma_commit(accf_bar(buf));
        }
      }
      if (!ok) {
        set_device_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
        if (issued) {
          // wait for the MMAs already issued before TMEM is freed
          ptx::mma_commit(drain_bar);
          const uint64_t grace = ptx::globaltimer_ns() + 100000000ull;
          while (!ptx::mbar_try_wait(drain_bar, 0u) && ptx::globaltimer_ns() < grace) {
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int ch_local = q * 32 + lane;
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total_units; u += gridDim.x, ++it) {
      const int buf = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      // one lane waits, the warp follows its verdict (tcgen05.ld below is
      // warp-collective, so the warp must agree)
      int got = 0;
      if (lane == 0) got = ptx::mbar_wait_bounded(accf_bar(buf), acc_phase, deadline, abort_flag) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const Unit x = decode_unit(u, offs, prefix, G, MT, S, BN);
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + 256u * buf;
      const int ch = x.mt * kBM + ch_local;
      const int n_mma = ((x.n_valid + 15) / 16) * 16;
      for (int c0 = 0; c0 < n_mma; c0 += 16) {
        uint32_t ra[16];
        ptx::tmem_ld16(taddr + c0, ra);
        if (MODE == kGateUp) {
          uint32_t rb[16];
          ptx::tmem_ld16(taddr + 128u + c0, rb);
          ptx::tmem_ld_wait();
          __nv_bfloat16* h = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < x.n_valid) {
              const float g = __uint_as_float(ra[j]);
              const float v = g / (1.f + __expf(-g)) * __uint_as_float(rb[j]);
              store_out(h + (size_t)(x.row0 + c0 + j) * p.M + ch, v);
            }
          }
        } else {
          ptx::tmem_ld_wait();
          if (p.out_f32) {
            float* y = static_cast<float*>(p.out) + (size_t)x.ks * p.R * p.M;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c0 + j < x.n_valid) y[(size_t)(x.row0 + c0 + j) * p.M + ch] = __uint_as_float(ra[j]);
          } else {
            __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c0 + j < x.n_valid) store_out(y + (size_t)(x.row0 + c0 + j) * p.M + ch, __uint_as_float(ra[j]));
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(acce_bar(buf));
    }
    if (!ok && lane == 0) set_device_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int MODE, int BN>
moe_status launch_one(const TcParams& p, const CUtensorMap& a0, const CUtensorMap& a1,
                      const CUtensorMap& b, int grid, cudaStream_t s) {
  using C = Cfg<MODE, BN>;
  auto kern = tc_grouped_kernel<MODE, BN>;
  MOE_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES));
  kern<<<grid, kThreads, C::SMEM_BYTES, s>>>(p, a0, a1, b);
  MOE_TRY_CUDA(cudaGetLastError());
  return MOE_OK;
}

template <int MODE>
moe_status launch_mode(int bn, const TcParams& p, const CUtensorMap& a0, const CUtensorMap& a1,
                       const CUtensorMap& b, int grid, cudaStream_t s) {
  if (bn == 32) return launch_one<MODE, 32>(p, a0, a1, b, grid, s);
  if (bn == 128) return launch_one<MODE, 128>(p, a0, a1, b, grid, s);
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace

TcPlan tc_plan(int T, int k, int E, int d, int ffn, int num_sms, int /*w_dtype*/) {
  TcPlan pl;
  const double R = (double)T * k;
  const double mean = R / E;
  const double est_max = mean + 3.0 * __builtin_sqrt(mean) + 1.0;
  pl.bn_gateup = est_max <= 32.0 ? 32 : 128;
  pl.bn_down = pl.bn_gateup;
  const double touched = E < R ? E : R;
  const double tiles_a = R / pl.bn_down;
  const int tiles = (int)(touched > tiles_a ? touched : tiles_a + 0.5);
  const int units = tiles * (d / kBM);
  const int kblocks = (ffn + kBK - 1) / kBK;
  pl.splits_down = 1;
  if (units < 2 * num_sms) {
    double best = 0.0;
    for (int s = 1; s <= 8; ++s) {
      if (kblocks / s < 4) break;
      const double u = (double)units * s;
      const double waves = __builtin_ceil(u / num_sms);
      const double eff = u / (waves * num_sms);
      if (eff > best + 0.02) {
        best = eff;
        pl.splits_down = s;
      }
    }
  }
  pl.grid = num_sms;
  return pl;
}

moe_status tc_grouped_launch(const TcGroupedArgs& a, const TcPlan& plan, cudaStream_t s,
                             cudaEvent_t mid) {
  if (a.R == 0) return MOE_OK;
  if (a.w_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (a.d % kBM != 0 || a.ffn % kBM != 0 || a.G > kMaxGroups) return MOE_ERR_UNSUPPORTED;
  CUtensorMap wg, wu, xb, wd, hb;
  MOE_TRY(make_tmap_2d(&wg, a.w_gate, (uint64_t)a.G * a.ffn, a.d, 2, kBM, kBK));
  MOE_TRY(make_tmap_2d(&wu, a.w_up, (uint64_t)a.G * a.ffn, a.d, 2, kBM, kBK));
  MOE_TRY(make_tmap_2d(&xb, a.x_perm, a.R, a.d, 2, kBoxN, kBK));
  MOE_TRY(make_tmap_2d(&wd, a.w_down, (uint64_t)a.G * a.d, a.ffn, 2, kBM, kBK));
  MOE_TRY(make_tmap_2d(&hb, a.h, a.R, a.ffn, 2, kBoxN, kBK));

  TcParams p{};
  p.G = a.G;
  p.offsets = a.offsets;
  p.R = a.R;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  p.selftest = 0;

  p.M = a.ffn;
  p.K = a.d;
  p.splits = 1;
  p.out = a.h;
  p.out_f32 = 0;
  MOE_TRY(launch_mode<kGateUp>(plan.bn_gateup, p, wg, wu, xb, plan.grid, s));
  if (mid != nullptr) MOE_TRY_CUDA(cudaEventRecord(mid, s));

  p.M = a.d;
  p.K = a.ffn;
  p.splits = plan.splits_down;
  p.out = a.y;
  p.out_f32 = plan.splits_down > 1 ? 1 : 0;
  MOE_TRY(launch_mode<kDown>(plan.bn_down, p, wd, wd, hb, plan.grid, s));
  return MOE_OK;
}

moe_status tc_selftest_launch(int* status, long long timeout_ns, cudaStream_t s) {
  CUtensorMap dummy;
  memset(&dummy, 0, sizeof(dummy));
  TcParams p{};
  p.G = 1;
  p.R = 0;
  p.M = kBM;
  p.K = kBK;
  p.splits = 1;
  p.status = status;
  p.timeout_ns = timeout_ns;
  p.selftest = 1;
  return launch_one<kGateUp, 32>(p, dummy, dummy, dummy, 1, s);
}

}  // namespace moe
