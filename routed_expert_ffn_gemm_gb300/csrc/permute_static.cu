// moe_permute_static_scratch: moe_permute for callers that cannot allocate
// device memory.
//
// Some callers have no way to hand this library a workspace: code hosted
// inside another framework whose memory manager must own every device
// allocation, or latency-critical loops where a cudaMalloc (which can
// synchronise the whole device) is not acceptable.  For them this entry point
// takes only the inputs and outputs of moe_permute and keeps the one piece of
// scratch the permutation needs -- the per-chunk expert counts of the large-
// batch path -- in a fixed array compiled into the library.
//
// The array is g_permute_scratch below: kStaticScratchInts int32 values
// (1 MiB).  Every GPU that loads the library holds it until the process
// exits.  Host code cannot use the array's name as a device address, so the
// first call on each device looks the address up with cudaGetSymbolAddress
// (with that device current) and caches it; that first call should therefore
// come before any stream capture.  The cached address does not survive a
// device reset (cudaDeviceReset) in the same process; neither does the rest
// of the library's per-device state.  All calls share the one array and it keeps
// the last call's contents; the count kernel overwrites every entry it later
// reads, so nothing has to be cleared between calls.  Calls whose work
// overlaps on the GPU (other streams, other threads) race on the array.
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

// ceil(T*k / 256) * E int32 counts must fit: e.g. T*k = 65536 with E <= 1024.
constexpr size_t kStaticScratchInts = 262144;

static __device__ __align__(256) int32_t g_permute_scratch[kStaticScratchInts];

constexpr int kMaxDevices = 64;
int32_t* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_permute_scratch on the current device (set-up once per
// device, with that device current).
moe_status static_scratch(int device, int32_t** out) {
  if (device < 0 || device >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[device] == nullptr) {
    void* p = nullptr;
    MOE_TRY_CUDA(cudaGetSymbolAddress(&p, g_permute_scratch));
    g_scratch_ptr[device] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[device];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_permute_static_scratch(const moe_problem* p, const int32_t* topk_idx,
                                                 const void* x, int32_t* counts, int32_t* offsets,
                                                 int32_t* perm_token, int32_t* inv_row,
                                                 void* x_perm, moe_stream_t stream) {
  using namespace moe;
  // the same problem checks as moe_permute, so both accept and refuse alike
  MOE_TRY(problem_check(p));
  if (counts == nullptr || offsets == nullptr || perm_token == nullptr || inv_row == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && topk_idx == nullptr) return MOE_ERR_INVALID_ARG;
  if ((x_perm != nullptr) != (x != nullptr)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(x_perm) & 15u))
    return MOE_ERR_INVALID_ARG;
  // the problem must fit the built-in scratch array
  const size_t need = permute_scratch_bytes(p->T, p->k, p->E);
  if (need > kStaticScratchInts * sizeof(int32_t)) {
    record_cuda_error_text("moe_permute_static_scratch: problem needs more than the 1 MiB built-in scratch");
    return MOE_ERR_WORKSPACE;
  }
  DeviceCtx ctx;
  MOE_TRY(device_ctx(&ctx));
  int32_t* scratch = nullptr;
  MOE_TRY(static_scratch(ctx.device, &scratch));
  const int act_bytes = p->act_dtype == MOE_F32 ? 4 : 2;
  PermuteArgs a{p->T, p->k, p->E, p->d, act_bytes, topk_idx, x, counts, offsets,
                perm_token, inv_row, x_perm, scratch, ctx.status};
  return permute_launch(a, reinterpret_cast<cudaStream_t>(stream));
}
