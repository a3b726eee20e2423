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
// Work unit = (expert g, tile of BN rows, channel tile mt, K split ks).
// A persistent grid (one CTA per SM) strides over the units; the per-expert
// tile counts are derived on the device from the offsets (no host sync).
// CTA roles (320 threads; 448 with converter warps):
//   warp 0 lane 0   TMA producer: weight tile(s) [128 x 64] + the row boxes
//                   per stage, 128-byte swizzle
//   warp 1 lane 0   MMA issuer: tcgen05.mma kind::f16, fp32 accumulate;
//                   warp 1 also allocates / frees 512 TMEM columns
//   warps 2..9      epilogue: tcgen05.ld from TMEM (two warps per lane
//                   quadrant, alternate column chunks), SiLU(g)*u (gate/up)
//                   or the projection (down), 64-byte coalesced stores
//   warps 10..13    (FP8 weights, f16 MMA) converters: E4M3 tile staged by TMA ->
//                   f16 tile, into tensor memory (decode tiles: the MMA
//                   reads A from TMEM) or into the 128-byte-swizzled
//                   shared-memory layout the MMA reads
// CTA pairs (prefill tiles): a cluster of two CTAs runs each unit with
// cta_group::2 MMAs, M = 256 channels (128 per CTA, each CTA's TMEM holding
// its own accumulator rows); each CTA stages its 128 weight rows and half
// of the unit's B rows, so per SM the B bytes per flop halve.  The even
// CTA issues the MMAs; the copies of both CTAs complete its barriers and
// its commits arrive on both CTAs' barriers.
// Accumulators live in TMEM (512 columns): a buffer holds the gate and up
// accumulators (gate at +0, up at +max(BN,128)) or the down accumulator;
// two buffers when they fit (BN <= 128 for gate/up, <= 256 for down), so the
// epilogue of one unit overlaps the next unit's loads and MMAs.  Every wait
// is bounded: on expiry the kernel records MOE_ERR_DEVICE_TIMEOUT, lets
// issued copies land, frees TMEM and returns.
//
// FP8 weights with bf16 activations ("MoE 推理部署", section 专家量化:
// per-expert scales): every bf16 row (token rows, rows of h) arrives as two
// E4M3 rows, hi and lo, with one power-of-two scale s per row and
// x = s * (hi + lo) -- the bf16 values themselves for every element within
// 2^9 of its row's largest magnitude (see the row split in quantize.cu).
// Both operands go straight from the TMA ring to tcgen05.mma kind::f8f6f4:
// each K step issues the MMA on the hi rows, then on the lo rows into the
// same accumulator, so one accumulator column per row holds W (hi + lo),
// and the epilogue multiplies it by s and the output channel's scale.  The
// products of E4M3 weights and E4M3 terms are exact, so this computes what
// a 16-bit MMA on the bf16 rows would, with no weight conversion.
// (The E4M3 -> f16 converter path below remains for MXFP4 weights, and for
// FP8 weights when MOE_FP8_CONVERT=1 selects it.)
//
// FP8 activations ("MOE推理流程解析", section 三: activations quantised
// before dispatch; gate/up only): the B rows arrive as E4M3 codes with one
// fp32 scale per token row, both operands go straight from the TMA ring to
// tcgen05.mma kind::f8f6f4 (K = 32 per instruction, 128-byte rows = 128
// elements of K per stage, no converter warps), and the epilogue multiplies
// each accumulator by its channel's weight scale and its column's row scale.
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <type_traits>

#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;          // output channels per tile (MMA M)
constexpr int kBK = 64;           // reduction elements per stage (128 bytes of bf16)
constexpr int kBoxSmall = 16;     // rows per B box for decode tiles (BN = 32)
constexpr int kBoxLarge = 128;    // rows per B box of the dense (router) GEMM
constexpr int kEpiWarps = 8;           // two per TMEM lane quadrant, alternating column chunks
constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer, MMA, epilogue warps
constexpr int kConvThreads = 128;      // FP8: 4 converter warps sharing each stage
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxGroups = 1024;
constexpr int kMaxGuSplits = 8;   // gate/up K splits (choose_splits and the override cap)
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
  const float* scale0;     // FP8: per-channel scales of A0 / A1 ([G*M])
  const float* scale1;
  int dense;               // 1: one group holding rows [0, R) (offsets unused)
  int boxn;                // rows per B box of tmB (16 or 64)
  // gate/up only, nullable: B row j of a group's tile is row
  // gather_rows[row0 + j] of tmB (the token rows, gathered by TMA gather4;
  // tmB's box is then one row high) instead of row row0 + j
  const int32_t* gather_rows;
  // gate/up K split with fused finalize (nullable): per (row tile, channel
  // tile) arrival counters, zero on entry and left zero; the CTA that
  // completes a tile's last split sums its partials in split order and
  // writes SiLU*mul to fin_out (bf16, or f16 with FP8 weights)
  int* tile_cnt;
  void* fin_out;
  // gate/up at prefill tiles (BN >= 128), with gather_rows: the producer
  // warp gathers the token rows from x_src itself with 16-byte cp.async
  // (row by row, 128-byte swizzle applied by hand) instead of reading a
  // materialised x_perm; the weights still come by TMA
  int lsu_gather;
  const void* x_src;
  int d_src;  // row length of x_src (elements)
  // two-term rows: rows between a row's hi codes and its lo codes in the B
  // matrix (the planes [2, rows, K] of the row split)
  int b_plane;
  // FP8 activations (gate/up): per-row quantisation scales of the B rows,
  // indexed by token (gather_rows) or by row
  const float* row_scale;
  // down GEMM, 1: the offsets and the weights were complete before the
  // predecessor grid passed its own griddepcontrol.wait (every grid between
  // their producer and this one lets dependants launch only after its
  // wait), so the unit walk and the first ring slots' weight copies start
  // before this grid's wait; only the B rows wait for the predecessor
  int early_w;
};

// Whether FP8 tiles take the tensor-memory operand path (see Cfg::TA): the
// decode tiles (32 rows) on single CTAs, and pair tiles whose accumulators
// (one buffer: gate and up of 128 rows, or the projection of up to 256)
// leave half of the 512 TMEM columns free.
__host__ __device__ constexpr bool ta_config(int mode, int bn, bool fp8, bool pair) {
  return fp8 && (pair ? (mode == kGateUp ? bn <= 128 : bn <= 256) : bn == 32);
}

// Weight formats of the kernel: bf16; FP8 weights converted to f16 for a
// kind::f16 MMA ("w8a16"); FP8 weights multiplied by FP8 token rows with a
// kind::f8f6f4 MMA (gate/up only: the FP8-activation mode); MXFP4 weights
// (E2M1 codes with a UE8M0 scale per 32 along K) converted to f16 for a
// kind::f16 MMA.
// FP8 weights times bf16 rows carried as two E4M3 terms (kind::f8f6f4,
// two B rows per row: the default for FP8 weights with bf16 activations).
// kWFp8X2W: the same with 256 elements of K per stage (two 128-byte K
// sub-tiles per operand), so that a stage carries twice the MMAs for its
// fixed costs (barrier waits, fences, commits).
enum { kWBf16 = 0, kWFp8 = 1, kWFp8Act8 = 2, kWMx4 = 3, kWFp8X2 = 4, kWFp8X2W = 5 };

template <int MODE, int BN, int WF, bool PAIR>
struct Cfg {
  static constexpr bool FP8 = WF != kWBf16;     // quantised weights: staged, f16 h (or E4M3 rows)
  static constexpr bool X2 = WF == kWFp8X2 || WF == kWFp8X2W;  // bf16 rows as two E4M3 rows
  static constexpr bool WIDE = WF == kWFp8X2W;  // 256 elements of K per stage each
  // E4M3 weights times E4M3 rows (kind::f8f6f4): FP8 activations, or the
  // two-term rows
  static constexpr bool A8 = WF == kWFp8Act8 || X2;
  static constexpr int NB = X2 ? 2 : 1;         // B tiles per stage: the hi rows, then the lo rows
  static constexpr bool H16 = FP8 && !X2;       // h stored in f16 (else bf16)
  static constexpr bool MX4 = WF == kWMx4;      // MXFP4 weights (block scales applied by the converters)
  static constexpr bool CHS = FP8 && !MX4;      // per-output-channel weight scales in the epilogue
  static constexpr bool CONV = WF == kWFp8 || MX4;  // converter warps write f16 weight operands
  // PAIR: a CTA pair (cluster of 2) runs one unit with cta_group::2 MMAs:
  // M = 256 output channels (128 per CTA, each CTA's TMEM holding its own
  // 128 accumulator rows for all N columns) and each CTA staging half of
  // the unit's B rows, so a CTA moves half the B bytes per flop
  static constexpr int CH = PAIR ? 2 * kBM : kBM;               // output channels per unit
  static constexpr int NA = MODE == kGateUp ? 2 : 1;           // weight operands per stage
  // FP8 tensor-memory operand path: the converters write the f16 weight
  // tile into tensor memory (tcgen05.st) and the MMA reads A from there, so
  // the f16 operand never passes through shared memory (whose bandwidth the
  // E4M3 tile, the f16 tile and the MMA's reads otherwise share).  Stages
  // span 128 elements of K: 128-byte E4M3 rows (64-byte rows cost as many
  // copy requests per row as 128-byte bf16 rows, for half the bytes), B in
  // two 64-element halves.
  static constexpr bool TA = ta_config(MODE, BN, CONV, PAIR);
  // bf16 down GEMM on pairs: 128 elements of K per stage as well, A and B
  // each in ONE copy (3-D boxes of two 64-element column blocks): half the
  // copies and half the barrier round trips per byte of a 64-element stage
  static constexpr bool K2 = MODE == kDown && PAIR && !FP8;     // (bf16 weights only)
  // FP8 activations: 128 elements of K per stage too, in single 128-byte
  // rows for both operands (one sub-tile); kind::f8f6f4 takes K = 32 per
  // instruction
  static constexpr int KB = WIDE ? 4 * kBK : TA || K2 || A8 ? 2 * kBK : kBK;  // K elements per stage
  static constexpr int SUBK = A8 ? 2 * kBK : kBK;              // K elements per 128-byte sub-tile
  static constexpr int NSUB = KB / SUBK;                       // 128-byte sub-tiles per operand and stage
  static constexpr int KSTEP = A8 ? 32 : 16;                   // K per MMA instruction
  static constexpr int A_BYTES = kBM * kBK * 2;                // 16 KB bf16 tile (MMA operand)
  static constexpr int BSUB_BYTES = (PAIR ? BN / 2 : BN) * kBK * 2;
  static constexpr int B_BYTES = NB * NSUB * BSUB_BYTES;
  // staged weight codes: E4M3 (8 or 16 KB), or packed E2M1 (half that)
  // followed by the UE8M0 block scales, KB/32 runs of 128 bytes
  static constexpr int STG_BYTES = FP8 ? (MX4 ? kBM * KB / 2 : kBM * KB) : 0;
  static constexpr int SCL_BYTES = MX4 ? KB / 32 * kBM : 0;
  // bf16: one ring of TMA slots [A0 A1 | B] read by the MMA.  FP8: a deep
  // ring of TMA slots [E4M3 A0 A1 | B] (cheap bytes: it hides HBM latency)
  // and a short ring of OSTAGES f16 operand slots [A0 A1] that the
  // converters fill and the MMA reads.
  // operand slots: enough that converters run ahead of the MMA's commits
  // (a commit round trip per slot otherwise serialises decode), while the
  // TMA ring keeps at least 4 slots
  static constexpr int OPND_BYTES = TA || !CONV ? 0 : NA * A_BYTES;
  static constexpr int W_BYTES_ = FP8 ? STG_BYTES + SCL_BYTES : NSUB * A_BYTES;
  static constexpr int SLOT_ = NA * W_BYTES_ + B_BYTES;
  static constexpr int AVAIL_ = kSmemLimit - 1024 - (8 * 40 + 16 + 4 * 2 * (kMaxGroups + 8));
  // TMEM: one accumulator buffer = NA accumulators of max(BN,128) columns;
  // two buffers when they fit beside the operand slots of the TA path
  static constexpr int UP_OFF = BN > 128 ? BN : 128;
  static constexpr int ACC_COLS = NA * UP_OFF;
  static constexpr bool TA_DECODE = TA && BN == 32;
  static constexpr int NBUF = TA && !TA_DECODE ? (2 * ACC_COLS + 2 * 64 * NA <= 512 ? 2 : 1)
                                               : (2 * ACC_COLS <= 512 ? 2 : 1);
  // TA operand slots of 64 columns (128 f16 of K per lane) per weight matrix
  static constexpr int TA_SLOTS = TA_DECODE ? 4 : (512 - NBUF * ACC_COLS) / 64;
  static constexpr int OSTAGES = !CONV ? 0 : TA ? (TA_SLOTS / NA > 4 ? 4 : TA_SLOTS / NA)
                                 : (AVAIL_ - 6 * SLOT_) / (NA * A_BYTES) >= 4 ? 4
                                 : (AVAIL_ - 6 * SLOT_) / (NA * A_BYTES) >= 3 ? 3 : 2;
  static constexpr int RING_OFF = OSTAGES * OPND_BYTES;
  static constexpr int W_BYTES = W_BYTES_;                      // weight tile bytes in a TMA slot
  // distance between the A matrices where the MMA reads them (TMA slot, or
  // FP8 operand slot)
  static constexpr int A_STRIDE = CONV ? A_BYTES : W_BYTES;
  static constexpr int B_OFF = (NA * W_BYTES + 1023) / 1024 * 1024;  // B keeps the 128-byte swizzle's alignment
  static constexpr int STAGE_BYTES = B_OFF + B_BYTES;           // multiple of 1024
  static constexpr int THREADS = kThreads + (CONV ? kConvThreads : 0);
  static constexpr int TAIL_BYTES = 8 * 40 + 16 + 4 * 2 * (kMaxGroups + 8);
  static constexpr int STAGES_FIT = (kSmemLimit - 1024 - TAIL_BYTES - RING_OFF) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 10 ? 10 : STAGES_FIT;
  static constexpr int BAR_OFF = RING_OFF + STAGES * STAGE_BYTES;
  // barriers: full[S], empty[S], opnd_full[4], opnd_empty[4], acc_full[2],
  // acc_empty[2], drain, rows_full[S] (gathered B rows of a pair CTA)
  static constexpr int NBARS = 3 * STAGES + 13;
  static constexpr int SLOT_OFF = BAR_OFF + 8 * NBARS;         // TMEM base address
  static constexpr int ABORT_OFF = SLOT_OFF + 8;
  static constexpr int OFFS_OFF = ABORT_OFF + 8;               // int offs[G+1]
  static constexpr int PREFIX_OFF = OFFS_OFF + 4 * (kMaxGroups + 4);
  static constexpr int SMEM_BYTES = PREFIX_OFF + 4 * (kMaxGroups + 4) + 1024;
  static_assert(STAGES >= 2, "pipeline too shallow");
  static_assert(SMEM_BYTES <= kSmemLimit, "shared memory budget");
  // At most one CTA of this kernel (of any instantiation) per SM: every CTA
  // takes all 512 TMEM columns before griddepcontrol.wait, and a second
  // co-resident CTA (a launch overlapped by programmatic dependence, or the
  // shared expert's kernel on the side stream) would block in tcgen05.alloc;
  // with CTA pairs, two clusters that each hold one SM of a TPC would wait
  // on each other for good.  Shared memory keeps them apart: two CTAs with
  // their 1 KB reservations overflow the SM's 228 KB.
  static_assert(2 * (SMEM_BYTES + 1024) > kSmemLimit + 1024, "one TMEM-holding CTA per SM");
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(BN % 16 == 0 && BN <= 256 && ACC_COLS <= 512, "tile rows");
  static_assert(!PAIR || BN >= 32, "pair tiles split B rows in halves");
  static_assert(!TA || (OSTAGES >= 2 && (TA_DECODE ? UP_OFF == 128 && ACC_COLS * NBUF <= 512 && OSTAGES * NA <= 4
                                                  : NBUF * ACC_COLS + OSTAGES * NA * 64 <= 512)),
                "TMEM operand slots");
  // TMEM column of operand slot o, weight matrix a (TA).  Decode tiles: the
  // 32-column accumulators sit at multiples of 128 and columns 64..127
  // after each hold an A tile; otherwise the A tiles follow the
  // accumulator buffers.
  static __device__ __forceinline__ uint32_t ta_col(int o, int a) {
    return TA_DECODE ? (uint32_t)(64 + 128 * (o * NA + a)) : (uint32_t)(NBUF * ACC_COLS + 64 * (o * NA + a));
  }
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

// SiLU(g) * u with SiLU(g) = g * sigmoid(g) and sigmoid(g) = (1 + tanh(g/2)) / 2:
// one hardware tanh (relative error ~2^-11, below the bf16 / f16 rounding
// of h) instead of an exponential and a division.
__device__ __forceinline__ float silu_mul(float g, float u) {
  const float a = 0.5f * g;
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(a));
  return fmaf(a, t, a) * u;
}

// Eight E4M3 values (two 32-bit words, lowest byte first) -> eight f16,
// exactly (every E4M3 value is representable in f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v16) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)v16));
  return h;
}

__device__ __forceinline__ uint4 e4m3x8_to_f16x8(uint32_t lo, uint32_t hi) {
  uint4 r;
  r.x = e4m3x2_to_f16x2(lo & 0xFFFFu);
  r.y = e4m3x2_to_f16x2(lo >> 16);
  r.z = e4m3x2_to_f16x2(hi & 0xFFFFu);
  r.w = e4m3x2_to_f16x2(hi >> 16);
  return r;
}

// MXFP4: the f16 pair multiplier 2^(s - 127) of a UE8M0 block scale s
// (exact f16 for s in [103, 142]: subnormal below 2^-14; the products
// code * 2^(s-127) are exact f16 values for s in [104, 140]).
__device__ __forceinline__ uint32_t ue8m0_to_f16x2(uint32_t s) {
  const int e = (int)s - 127;
  const uint32_t h = e >= -14 ? (e <= 15 ? (uint32_t)(e + 15) << 10 : 0x7C00u)
                              : (e >= -24 ? 1u << (e + 24) : 0u);
  return h | (h << 16);
}

// Eight E2M1 codes (one 32-bit word, element 2i in the low nibble of byte
// i) -> eight f16 (four pairs, the lower element in the low half), each
// times the block's multiplier m2: one hardware conversion per code pair
// (exact: every E2M1 value is an f16 value) and one f16x2 multiply by a
// power of two.
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t v, uint32_t m2, uint32_t* w) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .b32 h0, h1, h2, h3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 h0, b0;\n\tcvt.rn.f16x2.e2m1x2 h1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 h2, b2;\n\tcvt.rn.f16x2.e2m1x2 h3, b3;\n\t"
      "mul.rn.f16x2 %0, h0, %5;\n\tmul.rn.f16x2 %1, h1, %5;\n\t"
      "mul.rn.f16x2 %2, h2, %5;\n\tmul.rn.f16x2 %3, h3, %5;\n\t}"
      : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
      : "r"(v), "r"(m2));
}

// One 32-element MXFP4 block (16 bytes of codes) -> 32 f16 in w[0..15].
__device__ __forceinline__ void e2m1x32_to_f16(const uint4& v, uint32_t m2, uint32_t* w) {
  e2m1x8_to_f16x8(v.x, m2, w);
  e2m1x8_to_f16x8(v.y, m2, w + 4);
  e2m1x8_to_f16x8(v.z, m2, w + 8);
  e2m1x8_to_f16x8(v.w, m2, w + 12);
}

template <int MODE, int BN, int WF, bool PAIR>
__global__ void __launch_bounds__(Cfg<MODE, BN, WF, PAIR>::THREADS, 1)
    tc_grouped_kernel(const TcParams p, const __grid_constant__ CUtensorMap tmA0,
                      const __grid_constant__ CUtensorMap tmA1,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmS0,
                      const __grid_constant__ CUtensorMap tmS1) {
  // (tmS0 / tmS1: the MXFP4 block scales of A0 / A1; unused otherwise)
  using C = Cfg<MODE, BN, WF, PAIR>;
  constexpr bool FP8 = C::FP8, A8 = C::A8, CONV = C::CONV;
  constexpr int STAGES = C::STAGES;
  // pair barriers with remote arrivers live in the even CTA (rank 0)
  constexpr uint32_t kRemote = PAIR ? 2u : 1u;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = ptx::smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_s + pad;
  const uint32_t bars = sbase + C::BAR_OFF;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
  auto ofull_bar = [&](int c) { return bars + 8u * (2 * STAGES + c); };
  auto oempty_bar = [&](int c) { return bars + 8u * (2 * STAGES + 4 + c); };
  auto accf_bar = [&](int b) { return bars + 8u * (2 * STAGES + 8 + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (2 * STAGES + 10 + b); };
  const uint32_t drain_bar = bars + 8u * (2 * STAGES + 12);
  auto bfull_bar = [&](int s) { return bars + 8u * (2 * STAGES + 13 + s); };
  const bool lsu = MODE == kGateUp && p.lsu_gather != 0;
  // bf16 pairs gathering rows: each CTA's row copies complete its own
  // rows_full barrier; the odd CTA's MMA warp relays it to the even CTA
  const bool relay = PAIR && !CONV && lsu;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::SLOT_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::ABORT_OFF);
  int* offs = reinterpret_cast<int*>(smem + C::OFFS_OFF);
  int* prefix = reinterpret_cast<int*>(smem + C::PREFIX_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
  const bool leader = rank == 0u;
  // the even CTA's copy of a barrier (shared::cluster address)
  auto lead = [&](uint32_t bar) { return PAIR ? ptx::mapa_shared(bar, 0u) : bar; };
  // units: the pair walks one sequence together
  const int u_first = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int u_step = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  // weights and offsets ahead of the wait (down GEMM, no converter warps)
  const bool early = MODE == kDown && !CONV && p.early_w != 0 && !p.selftest && !p.dense;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // bf16 pairs: both producers arrive on the even CTA's full barrier
      // (their copies complete it); FP8: each CTA's converters wait on
      // their own CTA's copies
      // (+ 32 per-lane arrivals of the gathered rows, or the relayed
      // arrival of the odd CTA's rows)
      ptx::mbar_init(full_bar(s), PAIR && !CONV ? 2 + (relay ? 1 : 0) : 1 + (lsu ? 32 : 0));
      ptx::mbar_init(empty_bar(s), 1);
      ptx::mbar_init(bfull_bar(s), 32);
    }
    for (int c = 0; c < 4; ++c) {
      ptx::mbar_init(ofull_bar(c), kRemote * kConvThreads / 32);  // one arrival per converter warp
      ptx::mbar_init(oempty_bar(c), 1);                           // the MMA's commit
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(accf_bar(b), 1);
      ptx::mbar_init(acce_bar(b), kRemote * kEpiWarps);  // one arrival per epilogue warp
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0 && !p.selftest) {
    ptx::prefetch_tmap(&tmA0);
    if (MODE == kGateUp) ptx::prefetch_tmap(&tmA1);
    ptx::prefetch_tmap(&tmB);
    if (C::MX4) {
      ptx::prefetch_tmap(&tmS0);
      if (MODE == kGateUp) ptx::prefetch_tmap(&tmS1);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc<PAIR>(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish<PAIR>();
  }

  // The prologue above touches no global memory; from here on the previous
  // kernel's results (offsets, operands) must be complete.  Dependants may
  // launch once every CTA is past this wait, so a dependant that launches
  // knows every grid before this one has completed.
  if (!early) {
    griddep_wait();
    griddep_launch_dependents();
  }

  // Group row ranges (clamped into [0, R]) and the exclusive prefix of
  // per-group tile counts ceil(rows / BN).  (Early: read past L1, which
  // may hold lines of an earlier grid.)
  const int G = p.selftest ? 1 : p.G;
  for (int g = threadIdx.x; g <= G; g += C::THREADS) {
    int o = p.selftest ? 0 : (p.dense ? (g == 0 ? 0 : p.R) : early ? __ldcg(p.offsets + g) : p.offsets[g]);
    if (o < 0 || o > p.R) {
      set_device_status(p.status, MOE_ERR_DEVICE_BOUNDS);
      o = o < 0 ? 0 : p.R;
    }
    offs[g] = o;
  }
  __syncthreads();
  {
    const int per = (G + C::THREADS - 1) / C::THREADS;
    const int g0 = min(G, threadIdx.x * per), g1 = min(G, g0 + per);
    int local = 0;
    for (int g = g0; g < g1; ++g) local += (max(0, offs[g + 1] - offs[g]) + BN - 1) / BN;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    __shared__ int warp_sum[C::THREADS / 32];
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += warp_sum[w];
    int run = before + incl - local;
    for (int g = g0; g < g1; ++g) {
      prefix[g] = run;
      run += (max(0, offs[g + 1] - offs[g]) + BN - 1) / BN;
    }
    if (threadIdx.x == C::THREADS - 1) prefix[G] = before + incl;
  }
  ptx::tc_fence_before();
  // pairs: the peer's barriers must be initialised before any remote arrive
  if constexpr (PAIR)
    ptx::cluster_sync();
  else
    __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int MT = p.M / C::CH;
  const int S = p.splits;
  const int total_units = p.selftest ? 1 : prefix[G] * MT * S;
  const int kblocks = (p.K + C::KB - 1) / C::KB;
  const int kb_per_split = (kblocks + S - 1) / S;

  // Bytes one ring slot of unit x receives: the weight tiles and the B rows
  // (this CTA's half of them on a pair) of nbox boxes, or of nops gather4
  // copies; cp.async rows (lsu) arrive on their own.
  auto slot_bytes = [&](int nbox, int nops, bool gather_b) -> uint32_t {
    const uint32_t bbytes =
        lsu ? 0u : C::NB * C::NSUB * (gather_b ? (uint32_t)nops * 4 * kBK * 2 : (uint32_t)nbox * p.boxn * kBK * 2);
    return C::NA * C::W_BYTES + bbytes;
  };
  // Early weights: the first unit's first n_pre slots are armed with their
  // whole byte count and get their weight copies now; the producer adds
  // their B rows after the wait.  (The ring is empty: no slot to wait for.)
  int n_pre = 0;
  if (early) {
    if (warp == 0 && lane == 0 && u_first < total_units) {
      const Unit x = decode_unit(u_first, offs, prefix, G, MT, S, BN);
      // (the producer's weight policy below: evict-normal when several row
      // tiles of the expert read the weights)
      const uint64_t pol_w =
          prefix[x.g + 1] - prefix[x.g] > 1 ? ptx::policy_evict_normal() : ptx::policy_evict_first();
      const int kb0 = x.ks * kb_per_split, kb1 = min(kblocks, kb0 + kb_per_split);
      const int bhalf = PAIR ? ((x.n_valid + 31) / 32) * 16 : x.n_valid;
      const uint32_t bytes = slot_bytes((bhalf + p.boxn - 1) / p.boxn, 0, false);
      const int arow = x.g * p.M + x.mt * C::CH + (int)rank * kBM;
      n_pre = max(0, min(STAGES, kb1 - kb0));
      for (int i = 0; i < n_pre; ++i) {
        const int kb = kb0 + i;
        const uint32_t sa = sbase + C::RING_OFF + i * C::STAGE_BYTES;
        if (C::K2) {
          const uint32_t fb = lead(full_bar(i));
          ptx::mbar_arrive_expect_tx_cluster(fb, bytes);
          ptx::tma_load_3d_pair(sa, &tmA0, fb, arow, kb * 2, pol_w);
        } else if (PAIR) {
          const uint32_t fb = lead(full_bar(i));
          ptx::mbar_arrive_expect_tx_cluster(fb, bytes);
#pragma unroll
          for (int sub = 0; sub < (C::A8 ? C::NSUB : 1); ++sub)
            ptx::tma_load_2d_pair(sa + sub * (kBM * 128), &tmA0, fb, kb * C::KB + sub * C::SUBK, arow, pol_w);
        } else {
          ptx::mbar_arrive_expect_tx(full_bar(i), bytes);
#pragma unroll
          for (int sub = 0; sub < (C::A8 ? C::NSUB : 1); ++sub)
            ptx::tma_load_2d(sa + sub * (kBM * 128), &tmA0, full_bar(i), kb * C::KB + sub * C::SUBK, arow, pol_w);
        }
      }
    }
    griddep_wait();
    griddep_launch_dependents();
  }
  const uint64_t deadline = ptx::globaltimer_ns() + (uint64_t)p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Lane 0 waits for free slots and issues the weight copies and row
    // boxes; in gather mode the whole warp walks the units and every lane
    // issues up to two gather4 row copies per slot (otherwise lanes 1-31
    // leave at once: no warp-wide step per slot).
    const bool gather = p.gather_rows != nullptr && !lsu;
    if (!p.selftest && (gather || lsu || lane == 0)) {
      // weights: evict-first when one row tile of the expert reads them,
      // evict-normal when several do (they are read again while in L2)
      const uint64_t pol_w1 = ptx::policy_evict_first(), pol_wn = ptx::policy_evict_normal();
      const uint64_t pol_x = ptx::policy_evict_last();
      const uint32_t wmask = gather || lsu ? 0xffffffffu : 1u;
      // gathered rows: 16-bit elements (bf16 / f16), or E4M3 bytes (FP8 activations)
      const uint8_t* xs = static_cast<const uint8_t*>(p.x_src);
      constexpr int kEsz = A8 ? 1 : 2;
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;  // slots armed so far (the abort path derives their phases)
      bool ok = true;
      if (n_pre > 0) {
        // early slots (armed, their weights requested, before the wait):
        // the B rows of the first unit's first n_pre k-blocks
        const Unit x = decode_unit(u_first, offs, prefix, G, MT, S, BN);
        const int kb0 = x.ks * kb_per_split;
        const int bhalf = PAIR ? ((x.n_valid + 31) / 32) * 16 : x.n_valid;
        const int brow0 = x.row0 + (int)rank * bhalf;
        const int nbox = (bhalf + p.boxn - 1) / p.boxn;
        for (int i = 0; i < n_pre; ++i) {
          const int kb = kb0 + i;
          const uint32_t sb = sbase + C::RING_OFF + i * C::STAGE_BYTES + C::B_OFF;
          if (C::K2) {
            ptx::tma_load_3d_pair(sb, &tmB, lead(full_bar(i)), brow0, kb * 2, pol_x);
          } else {
#pragma unroll
            for (int term = 0; term < C::NB; ++term)
#pragma unroll
              for (int sub = 0; sub < C::NSUB; ++sub)
                for (int j = 0; j < nbox; ++j) {
                  const uint32_t dst = sb + (term * C::NSUB + sub) * C::BSUB_BYTES + j * p.boxn * kBK * 2;
                  const int kx = kb * C::KB + sub * C::SUBK, ry = brow0 + term * p.b_plane + j * p.boxn;
                  if (PAIR)
                    ptx::tma_load_2d_pair(dst, &tmB, lead(full_bar(i)), kx, ry, pol_x);
                  else
                    ptx::tma_load_2d(dst, &tmB, full_bar(i), kx, ry, pol_x);
                }
          }
        }
        stage = n_pre == STAGES ? 0 : n_pre;
        phase = n_pre == STAGES ? 1u : 0u;
        issued = n_pre;
      }
      for (int u = u_first; u < total_units && ok; u += u_step) {
        const Unit x = decode_unit(u, offs, prefix, G, MT, S, BN);
        const int kb0 = x.ks * kb_per_split, kb1 = min(kblocks, kb0 + kb_per_split);
        const uint64_t pol_w = prefix[x.g + 1] - prefix[x.g] > 1 ? pol_wn : pol_w1;
        // B rows this CTA stages: all of the tile, or (pair) its half of
        // the tile's MMA width rounded to 32
        const int bhalf = PAIR ? ((x.n_valid + 31) / 32) * 16 : x.n_valid;
        const int brow0 = x.row0 + (int)rank * bhalf;
        const int nbox = (bhalf + p.boxn - 1) / p.boxn;
        // gather4 copies of this tile: nops per B term (the hi rows, then,
        // two-term rows, the lo rows: rows of the lo plane, p.b_plane rows
        // further down the B matrix)
        const int nops = (x.n_valid + 3) / 4;
        // this lane's gather rows: ops lane and lane + 32 (NB * BN <= 256);
        // rows past the group's end repeat its first row (their columns are
        // unused)
        int gr[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int op = lane + 32 * h, term = op >= nops ? 1 : 0, i = 4 * (op - term * nops) + q;
            gr[h][q] = (gather && op < C::NB * nops)
                           ? p.gather_rows[x.row0 + (i < x.n_valid ? i : 0)] + term * p.b_plane
                           : 0;
          }
        // gathered rows (lsu): lanes 2j and 2j + 1 share rows j + 16 i of
        // the CTA's B rows; their token ids (-1: past the group's end, not
        // copied)
        constexpr int RPL = ((PAIR ? BN / 2 : BN) + 15) / 16;  // (80 rows on a 160-row pair tile: 5)
        int tok[RPL];
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
          const int rr = (lane >> 1) + 16 * i;
          const int r = brow0 + rr;
          tok[i] = (lsu && rr < bhalf && r < x.row0 + x.n_valid) ? p.gather_rows[r] : -1;
        }
        const uint32_t bytes = slot_bytes(nbox, nops, gather);
        const int arow = x.g * p.M + x.mt * C::CH + (int)rank * kBM;
        // (the first unit's early slots are already complete but for their B rows)
        for (int kb = u == u_first ? kb0 + n_pre : kb0; kb < kb1; ++kb) {
          int got = 1;
          if (lane == 0)
            got = ptx::mbar_wait_bounded(empty_bar(stage), phase ^ 1u, deadline, abort_flag) ? 1 : 0;
          if (gather || lsu) got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) {
            ok = false;
            break;
          }
          // weights: bf16 straight into the MMA tile, or E4M3 into staging
          const uint32_t sa = sbase + C::RING_OFF + stage * C::STAGE_BYTES;
          const uint32_t sb = sa + C::B_OFF;
          if (lane == 0) {
            ++issued;
            if (C::K2) {
              // one 3-D copy each for A and the B rows (two column blocks)
              const uint32_t fb = lead(full_bar(stage));
              ptx::mbar_arrive_expect_tx_cluster(fb, bytes);
              ptx::tma_load_3d_pair(sa, &tmA0, fb, arow, kb * 2, pol_w);
              ptx::tma_load_3d_pair(sb, &tmB, fb, brow0, kb * 2, pol_x);
            } else if (PAIR && !CONV) {
              // both CTAs' copies complete the even CTA's barrier
              const uint32_t fb = lead(full_bar(stage));
              ptx::mbar_arrive_expect_tx_cluster(fb, bytes);
#pragma unroll
              for (int sub = 0; sub < (C::A8 ? C::NSUB : 1); ++sub) {
                // (E4M3 weights: one 128-byte sub-tile of K per copy)
                const uint32_t so = sub * (kBM * 128);
                ptx::tma_load_2d_pair(sa + so, &tmA0, fb, kb * C::KB + sub * C::SUBK, arow, pol_w);
                if (MODE == kGateUp)
                  ptx::tma_load_2d_pair(sa + C::W_BYTES + so, &tmA1, fb, kb * C::KB + sub * C::SUBK, arow, pol_w);
              }
              if (!lsu)
#pragma unroll
                for (int term = 0; term < C::NB; ++term)
                  for (int i = 0; i < nbox; ++i)
#pragma unroll
                    for (int sub = 0; sub < C::NSUB; ++sub)
                      ptx::tma_load_2d_pair(sb + (term * C::NSUB + sub) * C::BSUB_BYTES + i * p.boxn * kBK * 2, &tmB,
                                            fb, kb * C::KB + sub * C::SUBK, brow0 + term * p.b_plane + i * p.boxn,
                                            pol_x);
            } else {
              ptx::mbar_arrive_expect_tx(full_bar(stage), bytes);
              // weight codes (MXFP4: two per byte), then (MXFP4) the
              // k-block's scales of the tile's 128 rows
              const int wx = C::MX4 ? kb * (C::KB / 2) : kb * C::KB;
#pragma unroll
              for (int sub = 0; sub < (C::A8 ? C::NSUB : 1); ++sub) {
                const uint32_t so = sub * (kBM * 128);
                ptx::tma_load_2d(sa + so, &tmA0, full_bar(stage), wx + sub * C::SUBK, arow, pol_w);
                if (MODE == kGateUp)
                  ptx::tma_load_2d(sa + C::W_BYTES + so, &tmA1, full_bar(stage), wx + sub * C::SUBK, arow, pol_w);
              }
              if constexpr (C::MX4) {
                const int sx = x.mt * C::CH + (int)rank * kBM, sy = x.g * (p.K / 32) + kb * (C::KB / 32);
                ptx::tma_load_2d(sa + C::STG_BYTES, &tmS0, full_bar(stage), sx, sy, pol_w);
                if (MODE == kGateUp)
                  ptx::tma_load_2d(sa + C::W_BYTES + C::STG_BYTES, &tmS1, full_bar(stage), sx, sy, pol_w);
              }
              if (!gather && !lsu)
#pragma unroll
                for (int term = 0; term < C::NB; ++term)
#pragma unroll
                  for (int sub = 0; sub < C::NSUB; ++sub)
                    for (int i = 0; i < nbox; ++i)
                      ptx::tma_load_2d(sb + (term * C::NSUB + sub) * C::BSUB_BYTES + i * p.boxn * kBK * 2, &tmB,
                                       full_bar(stage), kb * C::KB + sub * C::SUBK,
                                       brow0 + term * p.b_plane + i * p.boxn, pol_x);
            }
          }
          if (lsu) {
            // two lanes per row: of each 32-byte sector of the row's
            // 128-byte K slice (per 128-byte sub-tile) the even lane copies
            // the first 16 bytes and the odd lane the second, so that one
            // warp instruction asks for 16 whole sectors (one lane per row,
            // each 16-byte copy asking for half a sector, fetched every
            // sector twice); chunk c of row r goes to chunk c ^ (r % 8); then
            // one arrival per lane once its copies have landed
#pragma unroll
            for (int i = 0; i < RPL; ++i) {
              if (tok[i] < 0) continue;
              const int r = (lane >> 1) + 16 * i;
#pragma unroll
              for (int term = 0; term < C::NB; ++term)
#pragma unroll
                for (int sub = 0; sub < C::NSUB; ++sub) {
                  const uint8_t* src = xs + ((size_t)(tok[i] + term * p.b_plane) * p.d_src + (size_t)kb * C::KB +
                                             sub * C::SUBK) * kEsz;
                  const uint32_t dst = sb + (term * C::NSUB + sub) * C::BSUB_BYTES + r * 128;
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    const int c = 2 * j + (lane & 1);
                    ptx::cp_async16(dst + ((c ^ (r & 7)) << 4), src + 16 * c);
                  }
                }
            }
            ptx::cp_async_arrive_noinc(relay ? bfull_bar(stage) : full_bar(stage));
          }
          __syncwarp(wmask);
          if (gather) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int op = lane + 32 * h;
              const int term = op >= nops ? 1 : 0;
              if (op < C::NB * nops)
#pragma unroll
                for (int sub = 0; sub < C::NSUB; ++sub)
                  ptx::tma_gather4_2d(sb + (term * C::NSUB + sub) * C::BSUB_BYTES + (op - term * nops) * 4 * kBK * 2,
                                      &tmB, full_bar(stage), kb * C::KB + sub * C::SUBK, gr[h][0], gr[h][1], gr[h][2],
                                      gr[h][3], pol_x);
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && lsu) asm volatile("cp.async.wait_all;" ::: "memory");  // this lane's row copies
      if (!ok && lane == 0) {
        set_device_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
        // let every issued copy land before shared memory is released
        const uint64_t grace = ptx::globaltimer_ns() + 100000000ull;
        if (PAIR && !CONV && !leader) {
          // this CTA's copies complete the peer's barriers: wait a while
          const uint64_t t_end = ptx::globaltimer_ns() + 20000000ull;
          while (ptx::globaltimer_ns() < t_end) {
          }
        } else {
          // the last min(issued, STAGES) slots may still have copies in flight
          for (long long j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j) {
            const int s = (int)(j % STAGES);
            const uint32_t par = (uint32_t)((j / STAGES) & 1);
            while (!ptx::mbar_try_wait(full_bar(s), par) && ptx::globaltimer_ns() < grace) {
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (pairs: the even CTA issues for both)
    if (lane == 0 && leader) {
      bool ok = true;
      bool issued = false;
      // pairs: the commit arrives on the barrier at the same offset in both CTAs
      auto commit = [&](uint32_t bar) {
        if (PAIR)
          ptx::mma_commit_pair(bar);
        else
          ptx::mma_commit(bar);
      };
      if (p.selftest) {
        // nothing ever arrives on full_bar(0): the wait must expire
        ok = ptx::mbar_wait_bounded(full_bar(0), 0u, deadline, abort_flag);
      } else {
        int stage = 0, ostage = 0;
        uint32_t phase = 0, ophase = 0;
        int it = 0;
        for (int u = u_first; u < total_units && ok; u += u_step, ++it) {
          const Unit x = decode_unit(u, offs, prefix, G, MT, S, BN);
          const int kb0 = x.ks * kb_per_split, kb1 = min(kblocks, kb0 + kb_per_split);
          const int buf = it % C::NBUF;
          const uint32_t acc_phase = (uint32_t)(it / C::NBUF) & 1u;
          if (!ptx::mbar_wait_bounded(acce_bar(buf), acc_phase ^ 1u, deadline, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const int n_mma = PAIR ? ((x.n_valid + 31) / 32) * 32 : ((x.n_valid + 15) / 16) * 16;
          // (kind::f8f6f4 takes the same descriptor bits: E4M3 is format 0)
          const uint32_t idesc = FP8 ? ptx::idesc_f16_f32(C::CH, n_mma) : ptx::idesc_bf16_f32(C::CH, n_mma);
          const uint32_t d0 = tmem_base + (uint32_t)(C::ACC_COLS * buf);
          const uint32_t d1 = d0 + (uint32_t)C::UP_OFF;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!ptx::mbar_wait_bounded(full_bar(stage), phase, deadline, abort_flag) ||
                (relay && !ptx::mbar_wait_bounded(bfull_bar(stage), phase, deadline, abort_flag)) ||
                (CONV && !ptx::mbar_wait_bounded(ofull_bar(ostage), ophase, deadline, abort_flag))) {
              ok = false;
              break;
            }
            // rows gathered by cp.async are generic-proxy writes: order them
            // before the tensor core's reads
            if (lsu && !CONV) ptx::fence_proxy_async_smem();
            ptx::tc_fence_after();
            const uint32_t sa = sbase + C::RING_OFF + stage * C::STAGE_BYTES;
            const uint32_t aa = CONV ? sbase + ostage * C::OPND_BYTES : sa;
            const uint64_t da0 = ptx::sdesc_k_sw128(aa);
            const uint64_t da1 = ptx::sdesc_k_sw128(aa + C::A_STRIDE);
#pragma unroll
            for (int kk = 0; kk < C::KB / C::KSTEP; ++kk) {
              const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
              // B: 64-element sub-tile kk / 4, K step kk % 4 inside it
              const uint64_t db = ptx::sdesc_k_sw128(sa + C::B_OFF + (kk >> 2) * C::BSUB_BYTES) + 2 * (kk & 3);
              // A (TMA or operand slot): sub-tile kk / 4 as well (64 K each)
              const uint64_t ka = (uint64_t)((kk >> 2) * (C::A_BYTES >> 4)) + 2 * (kk & 3);
              if (C::TA) {
                const uint32_t at = tmem_base + 8u * kk;  // 16 f16 of K = 8 columns
                if (PAIR) {
                  ptx::mma_f16_ta_pair(d0, at + C::ta_col(ostage, 0), db, idesc, acc);
                  if (MODE == kGateUp) ptx::mma_f16_ta_pair(d1, at + C::ta_col(ostage, 1), db, idesc, acc);
                } else {
                  ptx::mma_f16_ta(d0, at + C::ta_col(ostage, 0), db, idesc, acc);
                  if (MODE == kGateUp) ptx::mma_f16_ta(d1, at + C::ta_col(ostage, 1), db, idesc, acc);
                }
              } else if (A8) {
                // E4M3 x E4M3: K = 32 per instruction, 32 bytes per step;
                // two-term rows: the hi tile, then the lo tile into the same
                // accumulator
#pragma unroll
                for (int term = 0; term < C::NB; ++term) {
                  const uint64_t dbt = db + (uint64_t)(term * ((C::NSUB * C::BSUB_BYTES) >> 4));
                  const uint32_t at = term > 0 ? 1u : acc;
                  if (PAIR) {
                    ptx::mma_f8_pair(d0, da0 + ka, dbt, idesc, at);
                    if (MODE == kGateUp) ptx::mma_f8_pair(d1, da1 + ka, dbt, idesc, at);
                  } else {
                    ptx::mma_f8(d0, da0 + ka, dbt, idesc, at);
                    if (MODE == kGateUp) ptx::mma_f8(d1, da1 + ka, dbt, idesc, at);
                  }
                }
              } else if (PAIR) {
                ptx::mma_f16_pair(d0, da0 + ka, db, idesc, acc);
                if (MODE == kGateUp) ptx::mma_f16_pair(d1, da1 + ka, db, idesc, acc);
              } else {
                ptx::mma_f16(d0, da0 + ka, db, idesc, acc);
                if (MODE == kGateUp) ptx::mma_f16(d1, da1 + ka, db, idesc, acc);
              }
            }
            issued = true;
            commit(empty_bar(stage));
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            if (CONV) {
              commit(oempty_bar(ostage));
              if (++ostage == C::OSTAGES) {
                ostage = 0;
                ophase ^= 1u;
              }
            }
          }
          if (ok) commit(accf_bar(buf));
        }
      }
      if (!ok) {
        set_device_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
        if (issued) {
          // wait for the MMAs already issued before TMEM is freed
          commit(drain_bar);
          const uint64_t grace = ptx::globaltimer_ns() + 100000000ull;
          while (!ptx::mbar_try_wait(drain_bar, 0u) && ptx::globaltimer_ns() < grace) {
          }
        }
      }
    }
    if (lane == 0 && !leader && relay && !p.selftest) {
      // odd CTA of a pair gathering rows: once this CTA's rows of a slot
      // have landed, make them visible to the tensor core and tell the
      // even CTA (its full barrier counts this arrival)
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = u_first; u < total_units && ok; u += u_step) {
        const Unit x = decode_unit(u, offs, prefix, G, MT, S, BN);
        const int kb0 = x.ks * kb_per_split, kb1 = min(kblocks, kb0 + kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait_bounded(bfull_bar(stage), phase, deadline, abort_flag)) {
            ok = false;
            break;
          }
          ptx::fence_proxy_async_smem();
          ptx::mbar_arrive_cluster(lead(full_bar(stage)));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) set_device_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
    }
  } else if (warp < kThreads / 32) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int ch_local = q * 32 + lane;
    const int eg = (warp - 2) >> 2;  // which of the quadrant's two warps: alternate column chunks
    int it = 0;
    bool ok = true;
    constexpr int CW = MODE == kGateUp ? 16 : 32;
    for (int u = u_first; u < total_units; u += u_step, ++it) {
      const int buf = it % C::NBUF;
      const uint32_t acc_phase = (uint32_t)(it / C::NBUF) & 1u;
      const Unit x = decode_unit(u, offs, prefix, G, MT, S, BN);
      // Every scale the unit's epilogue needs is requested before the
      // accumulator wait, so its memory latency hides behind the unit's MMAs.
      // E4M3 rows: for this warp's chunk i, lane l holds the row scale of the
      // chunk's column l (its row's scale; rows gathered by token: the token's).
      auto row_scale_of = [&](int cbase) -> float {
        const int c = cbase + lane;
        if (!A8 || lane >= CW || c >= x.n_valid) return 1.f;
        const int r = x.row0 + c;
        return __ldg(p.row_scale + (p.gather_rows != nullptr ? __ldg(p.gather_rows + r) : r));
      };
      constexpr int NCH = (BN + 2 * CW - 1) / (2 * CW);  // chunks per warp
      float rsv[NCH];
#pragma unroll
      for (int i = 0; i < NCH; ++i) rsv[i] = row_scale_of(eg * CW + 2 * CW * i);
      const int ch = x.mt * C::CH + (int)rank * kBM + ch_local;
      const float sc0 = C::CHS ? __ldg(p.scale0 + (size_t)x.g * p.M + ch) : 1.f;
      const float sc1 = C::CHS && MODE == kGateUp ? __ldg(p.scale1 + (size_t)x.g * p.M + ch) : 1.f;
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
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(C::ACC_COLS * buf);
      const bool empty_k = x.ks * kb_per_split >= kblocks;
      const int n_mma = ((x.n_valid + 15) / 16) * 16;
      // (not for 256-row tiles with converter warps, whose register cap is lower)
      if constexpr (MODE == kGateUp && !(C::CONV && BN > 160)) {
        if (!p.out_f32) {
          // h of every chunk is computed and packed into registers first, the
          // accumulator goes back to the MMA warp, and only then are the rows
          // stored: with one accumulator buffer the next unit's MMAs wait for
          // the release, not for the stores
          uint32_t hp[NCH][8];
#pragma unroll
          for (int i = 0; i < NCH; ++i) {
            const int c0 = eg * CW + 2 * CW * i;
            if (c0 < n_mma) {
              uint32_t ra[16], rb_[16];
              ptx::tmem_ld16(taddr + c0, ra);
              ptx::tmem_ld16(taddr + (uint32_t)C::UP_OFF + c0, rb_);
              ptx::tmem_ld_wait();
              if (empty_k) {
#pragma unroll
                for (int j = 0; j < 16; ++j) ra[j] = rb_[j] = 0u;
              }
#pragma unroll
              for (int j = 0; j < 16; j += 2) {
                const float r0 = A8 ? __shfl_sync(0xffffffffu, rsv[i], j) : 1.f;
                const float r1 = A8 ? __shfl_sync(0xffffffffu, rsv[i], j + 1) : 1.f;
                const float h0 = silu_mul(__uint_as_float(ra[j]) * sc0 * r0, __uint_as_float(rb_[j]) * sc1 * r0);
                const float h1 = silu_mul(__uint_as_float(ra[j + 1]) * sc0 * r1, __uint_as_float(rb_[j + 1]) * sc1 * r1);
                if (C::H16) {
                  const __half2 v = __floats2half2_rn(h0, h1);
                  hp[i][j / 2] = *reinterpret_cast<const uint32_t*>(&v);
                } else {
                  const __nv_bfloat162 v = __floats2bfloat162_rn(h0, h1);
                  hp[i][j / 2] = *reinterpret_cast<const uint32_t*>(&v);
                }
              }
            }
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (PAIR)
              ptx::mbar_arrive_cluster(lead(acce_bar(buf)));
            else
              ptx::mbar_arrive(acce_bar(buf));
          }
          // h is 16-bit either way (bf16, or f16 when it feeds an f16 MMA)
          uint16_t* o = static_cast<uint16_t*>(p.out) + (size_t)x.row0 * p.M + ch;
#pragma unroll
          for (int i = 0; i < NCH; ++i) {
            const int c0 = eg * CW + 2 * CW * i;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c0 + j < x.n_valid) o[(size_t)(c0 + j) * p.M] = (uint16_t)(hp[i][j / 2] >> (16 * (j & 1)));
          }
          continue;
        }
      }
      // CW accumulator columns per TMEM wait: 32 for the projection (its
      // epilogue is the longer one per MMA cycle), 16 for gate/up (measured
      // faster there).  BN is a multiple of 32, so columns past n_mma stay
      // inside this accumulator; they are not stored.
#pragma unroll 1
      for (int c0 = eg * CW; c0 < n_mma; c0 += 2 * CW) {
        const float rs_cur = rsv[0];
#pragma unroll
        for (int i = 0; i + 1 < NCH; ++i) rsv[i] = rsv[i + 1];
        uint32_t ra[CW], rb_[CW];
#pragma unroll
        for (int hlf = 0; hlf < CW / 16; ++hlf) {
          ptx::tmem_ld16(taddr + c0 + 16 * hlf, *reinterpret_cast<uint32_t(*)[16]>(&ra[16 * hlf]));
          if (MODE == kGateUp)
            ptx::tmem_ld16(taddr + (uint32_t)C::UP_OFF + c0 + 16 * hlf,
                           *reinterpret_cast<uint32_t(*)[16]>(&rb_[16 * hlf]));
        }
        ptx::tmem_ld_wait();
        if (empty_k) {
          // a K split past the end of K (ceil-sized splits): no MMA wrote
          // this accumulator, its partial sums are zero
#pragma unroll
          for (int j = 0; j < CW; ++j) ra[j] = rb_[j] = 0u;
        }
        // halves of 16 columns; the empty asm keeps the compiler from
        // interleaving them (which costs registers, not time)
#pragma unroll
        for (int hlf = 0; hlf < CW / 16; ++hlf) {
          // 16 accumulator columns: rows rb .. rb + NJ - 1 of the tile
          constexpr int NJ = 16;
          const int rb = c0 + 16 * hlf;
          const int nj = min(NJ, x.n_valid - rb);
          const uint32_t* a = ra + 16 * hlf;
          const uint32_t* b = rb_ + 16 * hlf;
          auto val = [&](const uint32_t* acc, int j) { return __uint_as_float(acc[j]); };
          if (nj > 0) {
            // E4M3 rows: each column (token row, or row of h) carries its
            // row's scale, from the lane that loaded it
            float rsc[NJ];
#pragma unroll
            for (int j = 0; j < NJ; ++j) rsc[j] = A8 ? __shfl_sync(0xffffffffu, rs_cur, 16 * hlf + j) : 1.f;
            if (MODE == kGateUp) {
              if (p.out_f32) {
                // K-split: scaled fp32 partials, SiLU*mul after the in-order sum
                float* row = static_cast<float*>(p.out) + ((size_t)x.ks * p.R + x.row0 + rb) * 2 * p.M + ch;
#pragma unroll
                for (int j = 0; j < NJ; ++j, row += 2 * p.M)
                  if (j < nj) {
                    row[0] = val(a, j) * sc0 * rsc[j];
                    row[p.M] = val(b, j) * sc1 * rsc[j];
                  }
              } else if (C::H16) {
                __half* o = static_cast<__half*>(p.out) + (size_t)(x.row0 + rb) * p.M + ch;  // h feeds an f16 MMA
#pragma unroll
                for (int j = 0; j < NJ; ++j, o += p.M)
                  if (j < nj) {
                    const float g = val(a, j) * sc0 * rsc[j];
                    *o = __float2half_rn(silu_mul(g, val(b, j) * sc1 * rsc[j]));
                  }
              } else {
                __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + (size_t)(x.row0 + rb) * p.M + ch;
#pragma unroll
                for (int j = 0; j < NJ; ++j, o += p.M)
                  if (j < nj) {
                    const float g = val(a, j) * sc0 * rsc[j];
                    store_out(o, silu_mul(g, val(b, j) * sc1 * rsc[j]));
                  }
              }
            } else if (p.out_f32) {
              float* o = static_cast<float*>(p.out) + ((size_t)x.ks * p.R + x.row0 + rb) * p.M + ch;
#pragma unroll
              for (int j = 0; j < NJ; ++j, o += p.M)
                if (j < nj) *o = val(a, j) * sc0 * rsc[j];
            } else {
              __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + (size_t)(x.row0 + rb) * p.M + ch;
#pragma unroll
              for (int j = 0; j < NJ; ++j, o += p.M)
                if (j < nj) store_out(o, val(a, j) * sc0 * rsc[j]);
            }
          }
          asm volatile("" ::: "memory");
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)
          ptx::mbar_arrive_cluster(lead(acce_bar(buf)));
        else
          ptx::mbar_arrive(acce_bar(buf));
      }
      if (MODE == kGateUp && p.out_f32 && p.tile_cnt != nullptr) {
        // fused finalize, per (tile, lane quadrant): the two warps of the
        // quadrant in each of the S splits arrive once their partials are
        // written; the warp whose arrival completes the 2*S sums the 32
        // channels' partials in split order (as the separate finalize
        // would), applies SiLU*mul, and sets the counter back to zero.  No
        // warp waits for another, so no barrier can hang.
        __threadfence();
        __syncwarp();
        int* cnt = p.tile_cnt + (u / S) * (PAIR ? 8 : 4) + (int)rank * 4 + q;
        int last = 0;
        if (lane == 0) last = atomicAdd(cnt, 1) == 2 * S - 1 ? 1 : 0;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
          const int c = x.mt * C::CH + (int)rank * kBM + ch_local;
          const float* part = static_cast<const float*>(p.out);
          for (int r = x.row0; r < x.row0 + x.n_valid; ++r) {
            // all of a row's partials in flight at once, then summed in order
            float gs[kMaxGuSplits], us[kMaxGuSplits];
#pragma unroll
            for (int sp = 0; sp < kMaxGuSplits; ++sp) {
              const float* row = part + ((size_t)min(sp, S - 1) * p.R + r) * 2 * p.M;
              gs[sp] = sp < S ? __ldcg(row + c) : 0.f;
              us[sp] = sp < S ? __ldcg(row + p.M + c) : 0.f;
            }
            float g = 0.f, uv = 0.f;
#pragma unroll
            for (int sp = 0; sp < kMaxGuSplits; ++sp) {
              g += gs[sp];
              uv += us[sp];
            }
            const float hv = silu_mul(g, uv);
            if (C::H16)
              static_cast<__half*>(p.fin_out)[(size_t)r * p.M + c] = __float2half_rn(hv);
            else
              store_out(static_cast<__nv_bfloat16*>(p.fin_out) + (size_t)r * p.M + c, hv);
          }
          if (lane == 0) *cnt = 0;
        }
      }
    }
    if (!ok && lane == 0) set_device_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
  } else if (CONV && !p.selftest) {
    // ------------------------------------------------------------ converters
    // Same unit / k-block walk as the MMA issuer; the four converter warps
    // share each stage.  Per k-block: wait for the E4M3 tiles in the TMA
    // slot and for a free operand slot, write the f16 tiles (tensor memory
    // or a shared-memory operand slot), make the writes visible to the
    // tensor core, then arrive on opnd_full.  The MMA's commit frees both
    // slots.
    const int ct = threadIdx.x - kThreads;  // 0 .. kConvThreads-1
    int stage = 0, ostage = 0;
    uint32_t phase = 0, ophase = 0;
    bool ok = true;
    for (int u = u_first; u < total_units && ok; u += u_step) {
      const Unit x = decode_unit(u, offs, prefix, G, MT, S, BN);
      const int kb0 = x.ks * kb_per_split, kb1 = min(kblocks, kb0 + kb_per_split);
      for (int kb = kb0; kb < kb1; ++kb) {
        int got = 0;
        if (lane == 0)
          got = ptx::mbar_wait_bounded(full_bar(stage), phase, deadline, abort_flag) &&
                        ptx::mbar_wait_bounded(oempty_bar(ostage), ophase ^ 1u, deadline, abort_flag)
                    ? 1
                    : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        const uint8_t* st = smem + C::RING_OFF + stage * C::STAGE_BYTES;
        // rows gathered by cp.async (generic proxy) sit in this slot: make
        // them visible to the tensor core before the operand arrival
        if (lsu) ptx::fence_proxy_async_smem();
        if constexpr (C::TA) {
          // one weight row per thread: the row is this warp's TMEM lane
          // (quadrant warp % 4); the 128-byte staging rows carry the 128-byte
          // swizzle (16-byte chunk c of row r at chunk c ^ (r & 7)), so the
          // warp's 32 rows read conflict-free; each half row (64 E4M3) fills
          // 32 TMEM columns
          ptx::tc_fence_after();
          const int qd = warp & 3;
          const int r = qd * 32 + lane;
          if constexpr (C::MX4) {
            // MXFP4: 64-byte rows of packed codes under the 64-byte swizzle
            // (16-byte chunk c of row r at chunk c ^ ((r / 2) % 4): the
            // warp's rows read conflict-free); chunk c is the c-th
            // 32-element block, its scale at byte c * 128 + r after the codes
#pragma unroll
            for (int a = 0; a < C::NA; ++a) {
              const uint8_t* src = st + a * C::W_BYTES + r * (C::KB / 2);
              const uint8_t* scl = st + a * C::W_BYTES + C::STG_BYTES + r;
#pragma unroll
              for (int hf = 0; hf < C::KB / 64; ++hf) {
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                  const int blk = 2 * hf + c;
                  const uint4 v = *reinterpret_cast<const uint4*>(src + ((blk ^ ((r >> 1) & 3)) << 4));
                  e2m1x32_to_f16(v, ue8m0_to_f16x2(scl[blk * kBM]), w + 16 * c);
                }
                ptx::tmem_st32(tmem_base + ((uint32_t)(qd * 32) << 16) + C::ta_col(ostage, a) + 32 * hf, w);
              }
            }
          } else {
#pragma unroll
            for (int a = 0; a < C::NA; ++a) {
              const uint8_t* src = st + a * C::STG_BYTES + r * C::KB;
#pragma unroll
              for (int hf = 0; hf < C::KB / 64; ++hf) {
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                  const uint4 v = *reinterpret_cast<const uint4*>(src + (((4 * hf + c) ^ (r & 7)) << 4));
                  const uint4 lo = e4m3x8_to_f16x8(v.x, v.y), hi = e4m3x8_to_f16x8(v.z, v.w);
                  w[8 * c + 0] = lo.x;
                  w[8 * c + 1] = lo.y;
                  w[8 * c + 2] = lo.z;
                  w[8 * c + 3] = lo.w;
                  w[8 * c + 4] = hi.x;
                  w[8 * c + 5] = hi.y;
                  w[8 * c + 6] = hi.z;
                  w[8 * c + 7] = hi.w;
                }
                ptx::tmem_st32(tmem_base + ((uint32_t)(qd * 32) << 16) + C::ta_col(ostage, a) + 32 * hf, w);
              }
            }
          }
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
        } else {
          // the f16 tile goes to the swizzled shared-memory operand slot
          // (16-byte chunk j of row r at chunk position j ^ (r % 8))
          uint8_t* op = smem + ostage * C::OPND_BYTES;
          if constexpr (C::MX4) {
            // MXFP4: 32-byte rows of packed codes (unswizzled), one
            // 32-element block per step -> four 16-byte f16 chunks
#pragma unroll
            for (int a = 0; a < C::NA; ++a) {
              const uint8_t* src = st + a * C::W_BYTES;
              uint8_t* dst = op + a * C::A_BYTES;
#pragma unroll 2
              for (int i = ct; i < kBM * (kBK / 32); i += kConvThreads) {
                const int r = i >> 1, c = i & 1;
                const uint4 v = *reinterpret_cast<const uint4*>(src + r * (kBK / 2) + c * 16);
                uint32_t w[16];
                e2m1x32_to_f16(v, ue8m0_to_f16x2(src[C::STG_BYTES + c * kBM + r]), w);
                const int sw = r & 7;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  *reinterpret_cast<uint4*>(dst + r * 128 + (((4 * c + j) ^ sw) << 4)) =
                      make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
              }
            }
          } else {
#pragma unroll
            for (int a = 0; a < C::NA; ++a) {
              const uint8_t* src = st + a * C::STG_BYTES;
              uint8_t* dst = op + a * C::A_BYTES;
#pragma unroll
              for (int i = ct; i < kBM * kBK / 16; i += kConvThreads) {  // 16 E4M3 per chunk
                const int r = i >> 2, c = i & 3;
                const uint4 v = *reinterpret_cast<const uint4*>(src + r * kBK + c * 16);
                const int sw = r & 7;
                *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * c) ^ sw) << 4)) = e4m3x8_to_f16x8(v.x, v.y);
                *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * c + 1) ^ sw) << 4)) = e4m3x8_to_f16x8(v.z, v.w);
              }
            }
          }
          ptx::fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          if (PAIR)
            ptx::mbar_arrive_cluster(lead(ofull_bar(ostage)));
          else
            ptx::mbar_arrive(ofull_bar(ostage));
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if (++ostage == C::OSTAGES) {
          ostage = 0;
          ophase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) set_device_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
  }

  ptx::tc_fence_before();
  // pairs: neither CTA leaves (or frees TMEM) while its peer may still
  // write its barriers or the MMA read its shared memory
  if constexpr (PAIR)
    ptx::cluster_sync();
  else
    __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc<PAIR>(tmem_base, kTmemCols);
  }
}

template <int MODE, int BN, int WF, bool PAIR = false>
moe_status launch_one(const TcParams& p, const CUtensorMap& a0, const CUtensorMap& a1,
                      const CUtensorMap& b, const CUtensorMap& s0, const CUtensorMap& s1, int grid,
                      cudaStream_t s) {
  using C = Cfg<MODE, BN, WF, PAIR>;
  auto kern = tc_grouped_kernel<MODE, BN, WF, PAIR>;
  MOE_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES));
  if (PAIR) {
    // The grid is persistent: every pair must be resident at once, and not
    // every SM finds a partner (clusters stay inside a GPC), so take the
    // number of co-resident pairs from the occupancy query (per device).
    // (host threads may launch concurrently: each entry is written once,
    // with the same value by whichever thread gets there)
    static std::atomic<int> resident[64];
    int dev = 0;
    MOE_TRY_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    if (resident[dev].load(std::memory_order_relaxed) == 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(grid & ~1);
      cfg.blockDim = dim3(C::THREADS);
      cfg.dynamicSmemBytes = C::SMEM_BYTES;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = 2;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      int n = 0;
      MOE_TRY_CUDA(cudaOccupancyMaxActiveClusters(&n, kern, &cfg));
      resident[dev].store(n > 0 ? n : -1, std::memory_order_relaxed);
    }
    const int r = resident[dev].load(std::memory_order_relaxed);
    if (r < 0) return MOE_ERR_UNSUPPORTED;
    grid = min(grid & ~1, 2 * r);
  }
  MOE_TRY_CUDA(launch_kc(PAIR ? 2 : 1, kern, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, s, p, a0, a1, b, s0, s1));
  MOE_TRY_CUDA(cudaGetLastError());
  return MOE_OK;
}

// The kernel instantiations: (rows per tile, weight format, CTA pair).
// s0 / s1: the MXFP4 block-scale maps of A0 / A1 (any map otherwise).
template <int MODE>
moe_status launch_mode(int bn, int wf, bool pair, const TcParams& p, const CUtensorMap& a0,
                       const CUtensorMap& a1, const CUtensorMap& b, const CUtensorMap& s0,
                       const CUtensorMap& s1, int grid, cudaStream_t s) {
#define MOE_LAUNCH(BN_, WF_, PAIR_) \
  if (bn == BN_ && wf == WF_) return launch_one<MODE, BN_, WF_, PAIR_>(p, a0, a1, b, s0, s1, grid, s)
  // (256 elements of K per stage: CTA pairs, and gate/up tiles up to 160
  // rows, so that at least two stages fit in shared memory)
#define MOE_LAUNCH_WIDE(BN_)                                                                             \
  if constexpr (MODE == kDown || BN_ <= 160)                                                             \
    if (bn == BN_ && wf == kWFp8X2W) return launch_one<MODE, BN_, kWFp8X2W, true>(p, a0, a1, b, s0, s1, grid, s)
  if (pair) {
    if (p.M % (2 * kBM) != 0 || grid < 2) return MOE_ERR_UNSUPPORTED;
    MOE_LAUNCH(32, kWFp8, true);
    MOE_LAUNCH(128, kWFp8, true);
    MOE_LAUNCH(256, kWFp8, true);
    MOE_LAUNCH(32, kWMx4, true);
    MOE_LAUNCH(128, kWMx4, true);
    MOE_LAUNCH(256, kWMx4, true);
    MOE_LAUNCH(32, kWBf16, true);
    MOE_LAUNCH(128, kWBf16, true);
    MOE_LAUNCH(256, kWBf16, true);
    MOE_LAUNCH(32, kWFp8Act8, true);
    MOE_LAUNCH(128, kWFp8Act8, true);
    MOE_LAUNCH(256, kWFp8Act8, true);
    MOE_LAUNCH(32, kWFp8X2, true);
    MOE_LAUNCH(128, kWFp8X2, true);
    MOE_LAUNCH(160, kWFp8X2, true);
    MOE_LAUNCH(256, kWFp8X2, true);
    MOE_LAUNCH_WIDE(128);
    MOE_LAUNCH_WIDE(160);
    MOE_LAUNCH_WIDE(256);
    return MOE_ERR_UNSUPPORTED;
  }
  MOE_LAUNCH(32, kWFp8, false);
  MOE_LAUNCH(128, kWFp8, false);
  MOE_LAUNCH(256, kWFp8, false);
  MOE_LAUNCH(32, kWMx4, false);
  MOE_LAUNCH(128, kWMx4, false);
  MOE_LAUNCH(256, kWMx4, false);
  MOE_LAUNCH(32, kWBf16, false);
  MOE_LAUNCH(128, kWBf16, false);
  MOE_LAUNCH(256, kWBf16, false);
  MOE_LAUNCH(32, kWFp8Act8, false);
  MOE_LAUNCH(128, kWFp8Act8, false);
  MOE_LAUNCH(256, kWFp8Act8, false);
  MOE_LAUNCH(32, kWFp8X2, false);
  MOE_LAUNCH(128, kWFp8X2, false);
  MOE_LAUNCH(160, kWFp8X2, false);
  MOE_LAUNCH(256, kWFp8X2, false);
#undef MOE_LAUNCH_WIDE
#undef MOE_LAUNCH
  return MOE_ERR_UNSUPPORTED;
}

int env_int(const char* name) {
  const char* v = getenv(name);
  return v ? atoi(v) : 0;
}

// (160-row tiles exist for two-term rows only)
int bn_ok(int bn, bool x2) { return bn == 32 || bn == 128 || bn == 256 || (bn == 160 && x2) ? bn : 0; }

}  // namespace

bool fp8_two_term(int w_dtype) {
  // (read on every call, like the other tuning switches: the workspace
  // size and the launches must see the same setting)
  return w_dtype == MOE_FP8_E4M3 && env_int("MOE_FP8_CONVERT") != 1;
}

bool fp8_two_term_scattered(int w_dtype, const TcPlan& plan) {
  if (!fp8_two_term(w_dtype)) return false;
  // decode tiles on CTA pairs: the rows scattered to their permuted order
  // and loaded by tiles (the gather4 row copies serve single CTAs here)
  if (plan.bn_gateup < 128) return plan.pair_gateup != 0;
  // prefill tiles: gathered per token by the producer warp's row copies
  // (two lanes per row), which measured faster than writing each token's
  // two rows to its k permuted rows and loading tiles (DeepSeek-V3-shaped
  // T=4096: 2.671 -> 2.640 ms); MOE_X2_SCATTER=1 scatters them (tuning)
  return env_int("MOE_X2_SCATTER") == 1;
}

namespace {

// K splits (<= 8, each >= 4 k-blocks) so that `units` work units fill whole
// waves of the SMs when there are fewer than two waves of them.
int choose_splits(int units, int kblocks, int num_sms) {
  int best_s = 1;
  if (units >= 2 * num_sms) return 1;
  double best = 0.0;
  for (int s = 1; s <= 8; ++s) {
    if (kblocks / s < 4) break;
    const double u = (double)units * s;
    const double waves = __builtin_ceil(u / num_sms);
    const double eff = u / (waves * num_sms);
    if (eff > best + 0.02) {
      best = eff;
      best_s = s;
    }
  }
  return best_s;
}

// h[r, c] = SiLU(sum_s g[s][r][c]) * sum_s u[s][r][c] from the gate/up
// GEMM's fp32 partials [S][R][2M] (g at column c, u at M + c), s in order.
template <typename OutT>
__global__ void __launch_bounds__(256) swiglu_finalize_kernel(int R, int M, int S,
                                                              const float* __restrict__ part,
                                                              OutT* __restrict__ h) {
  griddep_begin();
  const size_t n = (size_t)R * M;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / M, c = i % M;
    float g = 0.f, u = 0.f;
    for (int s = 0; s < S; ++s) {
      const float* row = part + ((size_t)s * R + r) * 2 * M;
      g += row[c];
      u += row[M + c];
    }
    const float v = g / (1.f + __expf(-g)) * u;
    if constexpr (sizeof(OutT) == 2 && std::is_same<OutT, __half>::value)
      h[i] = __float2half_rn(v);
    else
      h[i] = __float2bfloat16_rn(v);
  }
}
// Rows per B box: 16 for decode tiles; else one box for all of a CTA's B
// rows (BN, or BN/2 on a CTA pair): every TMA copy costs a fixed overhead
// on top of its bytes, measured to matter at prefill (two 64-row boxes in
// place of one 128-row box measured 10 % slower on the DeepSeek-shaped down
// GEMM, whose groups hold about 128 rows, though the larger box fetches
// rows of the next group).  MOE_BOXN, MOE_BOXN_GATEUP, MOE_BOXN_DOWN =
// 32/64/128/256 override (tuning) where they divide the CTA's rows, so the
// last box of a tile never writes past its shared-memory tile.
int boxn_of(int bn, bool pair, const char* env_name) {
  if (bn < 128) return kBoxSmall;
  const int cap = pair ? bn / 2 : bn;
  const int e = env_int(env_name) ? env_int(env_name) : env_int("MOE_BOXN");
  if ((e == 32 || e == 64 || e == 128 || e == 256) && e <= cap) return e;
  return cap;
}

}  // namespace

// Rows per tile from the expected rows per expert: 32 for decode (a few rows
// each), else 128; at prefill (>= 128 rows per expert on average) both GEMMs
// take 256.
// Gate/up at 256 rows has one TMEM buffer (its epilogue is not overlapped
// with the next unit's MMAs), yet on CTA pairs it moves the fewest operand
// bytes per flop and measured fastest on GB300 (with the eight-warp
// epilogue).  MOE_BN_GATEUP / MOE_BN_DOWN override (tuning).
TcPlan tc_plan(int T, int k, int E, int d, int ffn, int num_sms, int w_dtype) {
  TcPlan pl;
  const double R = (double)T * k;
  const double mean = R / E;
  const double est_max = mean + 3.0 * __builtin_sqrt(mean) + 1.0;
  const int bn = est_max <= 32.0 ? 32 : 128;
  // Converted FP8 weights (and MXFP4) keep 128-row gate/up tiles: on CTA
  // pairs their accumulators leave room in TMEM for the f16 weight operand
  // (the TA path).  Two-term rows (FP8 weights, bf16 activations) share one
  // accumulator column per row and tile like bf16.
  const bool x2 = fp8_two_term(w_dtype);
  const bool conv = (w_dtype == MOE_FP8_E4M3 && !x2) || w_dtype == MOE_MXFP4;
  int bn_gu = (bn == 128 && mean >= 128.0 && !conv) ? 256 : bn;
  int bn_dn = (bn == 128 && mean >= 128.0) ? 256 : bn;
  // Two-term rows with groups of about 100 to 160 rows (the DeepSeek-V3
  // shape at 4096 tokens: 128 on average) take 160-row tiles on CTA pairs:
  // 80 rows per CTA hold nearly every group in one tile, and their smaller
  // shared-memory tiles leave room for more pipeline stages (4 instead of 3
  // in gate/up, 6 instead of 4 in down) of bytes the GEMM actually uses.
  if (x2 && bn == 128 && E > 1 && mean >= 96.0 && est_max <= 192.0) bn_gu = bn_dn = 160;
  pl.bn_gateup = bn_ok(env_int("MOE_BN_GATEUP"), x2) ? env_int("MOE_BN_GATEUP") : bn_gu;
  pl.bn_down = bn_ok(env_int("MOE_BN_DOWN"), x2) ? env_int("MOE_BN_DOWN") : bn_dn;
  const double touched = E < R ? E : R;
  auto tiles_of = [&](int bn_) {
    const double a = R / bn_;
    return (int)(touched > a ? touched : a + 0.5);
  };
  // CTA pairs.  MOE_PAIR=0 keeps single CTAs; MOE_PAIR=2 also runs every
  // decode tile on pairs.  By default the decode (32-row) tiles of the bf16
  // down GEMM take pairs when that needs no more K splits: measured 5-11 %
  // faster on the down GEMM (fewer, larger units); so do the gate/up decode
  // tiles on two-term rows when their pair units need no K split (2.6 %
  // faster at 64 tokens of the DeepSeek-V3 shape; with K splits, at one
  // token, slower).  The other FP8 and FP8-activation decode tiles and the
  // bf16 gate/up decode tiles measured no faster on pairs (within 1-2 %).
  const char* pe = getenv("MOE_PAIR");
  const bool pairs_ok = !(pe != nullptr && pe[0] == '0') && num_sms >= 2;
  const bool act8 = w_dtype == MOE_FP8_E4M3_ACT8 || x2;  // (E4M3 rows: kind::f8f6f4)
  const bool fp8 = w_dtype == MOE_FP8_E4M3 || act8 || w_dtype == MOE_MXFP4;
  const bool dec_pairs = pairs_ok && pe != nullptr && pe[0] == '2';
  // K per stage: 128 on the FP8 tensor-memory operand path (decode tiles),
  // with E4M3 rows (128-byte rows of both operands), and for the bf16
  // down GEMM on pairs (two column blocks per copy)
  const int kw_dn = act8 || (fp8 && pl.bn_down == 32) ? 2 * kBK : kBK;
  const int kw_gu = act8 || (fp8 && pl.bn_gateup == 32) ? 2 * kBK : kBK;
  // K splits of single-CTA units, and of pair units (2 SMs each, 256
  // channels, 128 of K per stage)
  const int kb_dn = (ffn + kw_dn - 1) / kw_dn, kb_dn_pair = (ffn + 2 * kBK - 1) / (2 * kBK);
  const int s_dn = choose_splits(tiles_of(pl.bn_down) * (d / kBM), kb_dn, num_sms);
  const int s_dn_pair = choose_splits(tiles_of(pl.bn_down) * (d / (2 * kBM)), kb_dn_pair, num_sms / 2);
  const bool dn_pair_fits = pl.bn_down == 32 && d % (2 * kBM) == 0;
  const bool dec_pair_dn = dn_pair_fits && (dec_pairs || (pairs_ok && w_dtype == MOE_BF16 && s_dn_pair <= s_dn));
  const int s_gu_pair = choose_splits(tiles_of(pl.bn_gateup) * (ffn / (2 * kBM)), (d + 2 * kBK - 1) / (2 * kBK),
                                      num_sms / 2);
  const bool dec_pair_gu = pl.bn_gateup == 32 && ffn % (2 * kBM) == 0 &&
                           (dec_pairs || (pairs_ok && x2 && s_gu_pair == 1 && mean < 128.0));
  pl.splits_down = dec_pair_dn ? s_dn_pair : s_dn;
  pl.splits_gateup = dec_pair_gu
                         ? s_gu_pair
                         : choose_splits(tiles_of(pl.bn_gateup) * (ffn / kBM), (d + kw_gu - 1) / kw_gu, num_sms);
  // (no gate/up split for groups of prefill size: their tiles fill the SMs,
  // and a split adds a pass over fp32 partials of every row)
  if (mean >= 128.0) pl.splits_gateup = 1;
  if (env_int("MOE_SPLITS_GATEUP") >= 1 && env_int("MOE_SPLITS_GATEUP") <= 8)
    pl.splits_gateup = env_int("MOE_SPLITS_GATEUP");
  pl.grid = num_sms;
  // and pairs at prefill tiles (>= 128 rows) when the channel count splits
  // into 256-channel pair tiles
  pl.pair_gateup =
      dec_pair_gu || (pairs_ok && pl.bn_gateup >= 128 && ffn % (2 * kBM) == 0 && pl.splits_gateup == 1) ? 1 : 0;
  pl.pair_down = dec_pair_dn || (pairs_ok && pl.bn_down >= 128 && d % (2 * kBM) == 0) ? 1 : 0;
  pl.boxn_gateup = boxn_of(pl.bn_gateup, pl.pair_gateup != 0, "MOE_BOXN_GATEUP");
  pl.boxn_down = boxn_of(pl.bn_down, pl.pair_down != 0, "MOE_BOXN_DOWN");
  return pl;
}

moe_status tc_grouped_launch(const TcGroupedArgs& a, const TcPlan& plan, cudaStream_t s,
                             cudaEvent_t mid) {
  if (a.R == 0) return MOE_OK;
  const bool x2 = fp8_two_term(a.w_dtype);                     // bf16 rows as two E4M3 rows
  const int nb = x2 ? 2 : 1;                                   // planes of E4M3 rows (hi, lo)
  const bool fa8 = a.w_dtype == MOE_FP8_E4M3_ACT8;             // FP8 activations
  const bool act8 = fa8 || x2;                                 // E4M3 rows, kind::f8f6f4
  const bool mx4 = a.w_dtype == MOE_MXFP4;
  const bool fp8 = a.w_dtype == MOE_FP8_E4M3 || act8 || mx4;  // quantised weights
  const bool h16 = fp8 && !x2;                                 // h in f16 (converted weights, FP8 activations)
  if (!fp8 && a.w_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (fp8 && (a.s_gate == nullptr || a.s_up == nullptr || a.s_down == nullptr)) return MOE_ERR_INVALID_ARG;
  if (act8 && (a.row_scale == nullptr || a.h_q == nullptr || a.h_scale == nullptr)) return MOE_ERR_INVALID_ARG;
  const int wf_base = x2 ? kWFp8X2 : fa8 ? kWFp8Act8 : mx4 ? kWMx4 : fp8 ? kWFp8 : kWBf16;
  // two-term rows on CTA pairs at prefill tiles: 256 elements of K per
  // stage (MOE_X2_WIDE: bit 0 down, bit 1 gate/up)
  const int xw = getenv("MOE_X2_WIDE") != nullptr ? env_int("MOE_X2_WIDE") : 1;
  const bool wide_gu = x2 && plan.pair_gateup && plan.bn_gateup >= 128 && plan.bn_gateup <= 160 && (xw & 2);
  const bool wide_dn = x2 && plan.pair_down && plan.bn_down >= 128 && (xw & 1);
  const int wf_gu = wide_gu ? kWFp8X2W : wf_base;
  const int wf_dn = wide_dn ? kWFp8X2W : wf_base;
  if (a.d % kBM != 0 || a.ffn % kBM != 0 || a.G > kMaxGroups) return MOE_ERR_UNSUPPORTED;
  // weights: bf16 tiles [128 x 64] with 128-byte swizzle, or E4M3 tiles
  // [128 x 64 bytes] staged unswizzled for the converters
  const int wb = fp8 ? 1 : 2;
  // E4M3 staging for the tensor-memory operand path (decode tiles): boxes
  // 128 bytes wide with the 128-byte swizzle its converters read
  // conflict-free
  // FP8 activations: E4M3 weight and row tiles straight into the MMA's
  // 128-byte-swizzled operands, 128 elements of K per row
  // MXFP4: packed codes, half as many bytes per K: 64-byte rows under the
  // 64-byte swizzle (tensor-memory path, 128 of K) or 32-byte rows
  // unswizzled (64 of K); the block scales [G, K/32, M] as a 2-D byte
  // array [G*K/32, M], one box of (K per stage / 32) x 128 per tile
  const bool ta_gu = ta_config(kGateUp, plan.bn_gateup, fp8 && !act8, plan.pair_gateup != 0);
  const bool ta_dn = ta_config(kDown, plan.bn_down, fp8 && !act8, plan.pair_down != 0);
  const int wsw_gu = mx4 ? (ta_gu ? 64 : 0) : !fp8 || ta_gu || act8 ? 128 : 0;
  const int wsw_dn = mx4 ? (ta_dn ? 64 : 0) : !fp8 || ta_dn || act8 ? 128 : 0;
  const int kw_gu = ta_gu || act8 ? 2 * kBK : kBK, kw_dn = ta_dn || act8 ? 2 * kBK : kBK;  // K per stage
  const int wk_gu = mx4 ? kw_gu / 2 : kw_gu, wk_dn = mx4 ? kw_dn / 2 : kw_dn;    // box columns
  const uint64_t wcols_gu = mx4 ? a.d / 2 : a.d, wcols_dn = mx4 ? a.ffn / 2 : a.ffn;
  CUtensorMap wg, wu, xb, wd, hb, sg, su, sd;
  MOE_TRY(make_tmap_2d(&wg, a.w_gate, (uint64_t)a.G * a.ffn, wcols_gu, wb, kBM, wk_gu, wsw_gu));
  MOE_TRY(make_tmap_2d(&wu, a.w_up, (uint64_t)a.G * a.ffn, wcols_gu, wb, kBM, wk_gu, wsw_gu));
  if (mx4) {
    MOE_TRY(make_tmap_2d(&sg, a.s_gate, (uint64_t)a.G * (a.d / 32), a.ffn, 1, kw_gu / 32, kBM, 0));
    MOE_TRY(make_tmap_2d(&su, a.s_up, (uint64_t)a.G * (a.d / 32), a.ffn, 1, kw_gu / 32, kBM, 0));
    MOE_TRY(make_tmap_2d(&sd, a.s_down, (uint64_t)a.G * (a.ffn / 32), a.d, 1, kw_dn / 32, kBM, 0));
  } else {
    sg = su = sd = wg;
  }
  const int box_gu = plan.boxn_gateup > 0 ? plan.boxn_gateup : kBoxSmall;
  const int box_dn = plan.boxn_down > 0 ? plan.boxn_down : kBoxSmall;
  // gathered token rows: TMA gather4 for decode tiles, cp.async by the
  // producer warp for prefill tiles (gather4 costs a copy per 4 rows)
  const bool lsu = a.gather_rows != nullptr && (plan.bn_gateup >= 128 || plan.pair_gateup);
  if (plan.pair_gateup && a.gather_rows != nullptr && !lsu) return MOE_ERR_UNSUPPORTED;
  // row operand: 128-byte rows, 64 16-bit elements or 128 E4M3 codes
  // (two-term rows: two planes of code rows, hi then lo, one matrix)
  const int xe = act8 ? 1 : 2, xk = act8 ? 2 * kBK : kBK;
  if (a.gather_rows != nullptr)  // token rows by index: one-row boxes for gather4
    MOE_TRY(make_tmap_2d(&xb, a.x_src, (uint64_t)nb * a.T_src, a.d, xe, 1, xk, 128));
  else
    MOE_TRY(make_tmap_2d(&xb, a.x_perm, (uint64_t)nb * a.R, a.d, xe, box_gu, xk, 128));
  // bf16 down GEMM on pairs: 3-D maps, one copy per operand and stage (its
  // B rows in one box: all BN/2 rows of the CTA)
  const bool k2_dn = !fp8 && plan.pair_down;
  if (k2_dn) {
    MOE_TRY(make_tmap_kpair(&wd, a.w_down, (uint64_t)a.G * a.d, a.ffn, 2, kBM));
    MOE_TRY(make_tmap_kpair(&hb, a.h, a.R, a.ffn, 2, plan.bn_down / 2));
  } else {
    MOE_TRY(make_tmap_2d(&wd, a.w_down, (uint64_t)a.G * a.d, wcols_dn, wb, kBM, wk_dn, wsw_dn));
    // h rows: 16-bit, or their E4M3 codes (two planes for two-term rows), 128-byte rows
    if (act8)
      MOE_TRY(make_tmap_2d(&hb, a.h_q, (uint64_t)nb * a.R, a.ffn, 1, box_dn, 2 * kBK, 128));
    else
      MOE_TRY(make_tmap_2d(&hb, a.h, a.R, a.ffn, 2, box_dn, kBK, 128));
  }

  TcParams p{};
  p.G = a.G;
  p.offsets = a.offsets;
  p.R = a.R;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  p.selftest = 0;

  p.M = a.ffn;
  p.K = a.d;
  p.dense = a.offsets == nullptr ? 1 : 0;  // one group holding rows [0, R)
  const bool gu_split = plan.splits_gateup > 1 && a.gu_partials != nullptr;
  const bool gu_fused = gu_split && a.gu_cnt != nullptr;
  p.tile_cnt = gu_fused ? a.gu_cnt : nullptr;
  p.fin_out = gu_fused ? a.h : nullptr;
  p.splits = gu_split ? plan.splits_gateup : 1;
  p.out = gu_split ? static_cast<void*>(a.gu_partials) : a.h;
  p.out_f32 = gu_split ? 1 : 0;
  p.scale0 = a.s_gate;
  p.scale1 = a.s_up;
  p.boxn = box_gu;
  p.gather_rows = a.gather_rows;
  p.lsu_gather = lsu ? 1 : 0;
  p.x_src = a.x_src;
  p.d_src = a.d;
  p.b_plane = a.gather_rows != nullptr ? a.T_src : a.R;
  p.row_scale = act8 ? a.row_scale : nullptr;
  MOE_TRY(launch_mode<kGateUp>(plan.bn_gateup, wf_gu, plan.pair_gateup != 0, p, wg, wu, xb, sg, su, plan.grid, s));
  p.gather_rows = nullptr;
  p.lsu_gather = 0;
  p.row_scale = nullptr;
  p.tile_cnt = nullptr;
  p.fin_out = nullptr;
  if (gu_split && !gu_fused) {
    const size_t n = (size_t)a.R * a.ffn;
    const int blocks = (int)((n + 255) / 256 < 8192 ? (n + 255) / 256 : 8192);
    if (h16)
      MOE_TRY_CUDA(launch_k(swiglu_finalize_kernel<__half>, dim3(blocks), dim3(256), 0, s, a.R, a.ffn,
                            plan.splits_gateup, (const float*)a.gu_partials, static_cast<__half*>(a.h)));
    else
      MOE_TRY_CUDA(launch_k(swiglu_finalize_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, s, a.R,
                            a.ffn, plan.splits_gateup, (const float*)a.gu_partials,
                            static_cast<__nv_bfloat16*>(a.h)));
  }
  if (mid != nullptr) MOE_TRY_CUDA(record_event(mid, s));
  // FP8 activations: h's rows quantised per row for the down GEMM; two-term
  // rows: h's bf16 rows split exactly into their two E4M3 rows
  if (fa8) MOE_TRY(quantize_rows_e4m3_launch(a.h, a.R, a.ffn, a.h_q, a.h_scale, plan.grid, s, true));
  if (x2) MOE_TRY(split_rows_e4m3x2_launch(a.h, a.R, a.ffn, a.h_q, a.h_scale, plan.grid, s));

  p.M = a.d;
  p.K = a.ffn;
  p.b_plane = a.R;  // (two-term rows of h: planes [2, R, ffn])
  p.splits = plan.splits_down;
  p.out = a.y;
  p.out_f32 = plan.splits_down > 1 ? 1 : 0;
  p.scale0 = a.s_down;
  p.scale1 = nullptr;
  p.row_scale = act8 ? a.h_scale : nullptr;
  p.boxn = k2_dn ? plan.bn_down / 2 : box_dn;
  p.early_w = a.early_down;
  MOE_TRY(launch_mode<kDown>(plan.bn_down, wf_dn, plan.pair_down != 0, p, wd, wd, hb, sd, sd, plan.grid, s));
  return MOE_OK;
}

size_t gu_counters_size(int R, int G, int ffn, const TcPlan& plan) {
  if (plan.splits_gateup <= 1) return 0;
  const size_t tiles = (size_t)R / plan.bn_gateup + (size_t)G;  // sum of ceil(n_g / BN)
  const int ch = plan.pair_gateup ? 2 * kBM : kBM;
  return tiles * (size_t)(ffn / ch) * (plan.pair_gateup ? 8 : 4);  // per (tile, channel tile, CTA, quadrant)
}

moe_status tc_dense_f32_launch(const void* a, const void* b, float* out, int M, int N, int K,
                               int splits, int num_sms, int* status, long long timeout_ns,
                               cudaStream_t s) {
  if (N == 0) return MOE_OK;
  if (M % kBM != 0 || K % 8 != 0 || splits < 1) return MOE_ERR_UNSUPPORTED;
  CUtensorMap ta, tb;
  MOE_TRY(make_tmap_2d(&ta, a, (uint64_t)M, K, 2, kBM, kBK, 128));
  MOE_TRY(make_tmap_2d(&tb, b, (uint64_t)N, K, 2, kBoxLarge, kBK, 128));
  TcParams p{};
  p.G = 1;
  p.dense = 1;
  p.R = N;
  p.M = M;
  p.K = K;
  p.splits = splits;
  p.out = out;
  p.out_f32 = 1;
  p.status = status;
  p.timeout_ns = timeout_ns;
  p.boxn = kBoxLarge;
  return launch_mode<kDown>(128, kWBf16, false, p, ta, ta, tb, ta, ta, num_sms, s);
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
  p.boxn = kBoxSmall;
  return launch_one<kGateUp, 32, kWBf16>(p, dummy, dummy, dummy, dummy, dummy, 1, s);
}

}  // namespace moe
