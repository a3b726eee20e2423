// Library runtime: per-device context (SM count, kernel status word),
// CUDA error text, TMA tensor-map encoding, status strings.
#include <mutex>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"

namespace moe {

// The per-device kernel status word: 0 = no error, else the first
// moe_status a kernel recorded since the last moe_read_device_status().
__device__ int g_kernel_status;

namespace {

constexpr int kMaxDevices = 64;
DeviceCtx g_ctx[kMaxDevices];
std::mutex g_ctx_mu;

thread_local char g_last_error[256] = "";

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

}  // namespace

void record_cuda_error_text(const char* text) {
  strncpy(g_last_error, text, sizeof(g_last_error) - 1);
  g_last_error[sizeof(g_last_error) - 1] = 0;
}

void record_cuda_error(cudaError_t err) {
  record_cuda_error_text(cudaGetErrorString(err));
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("MOE_PDL");
    return !(v != nullptr && v[0] == '0');
  }();
  return on;
}

moe_status device_ctx(DeviceCtx* out) {
  int dev = -1;
  MOE_TRY_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_ctx_mu);
  DeviceCtx& c = g_ctx[dev];
  if (c.device != dev) {
    int sms = 0;
    MOE_TRY_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    void* p = nullptr;
    MOE_TRY_CUDA(cudaGetSymbolAddress(&p, g_kernel_status));
    c.num_sms = sms;
    c.status = static_cast<int*>(p);
    MOE_TRY_CUDA(cudaStreamCreateWithFlags(&c.side, cudaStreamNonBlocking));
    MOE_TRY_CUDA(cudaEventCreateWithFlags(&c.fork, cudaEventDisableTiming));
    MOE_TRY_CUDA(cudaEventCreateWithFlags(&c.join, cudaEventDisableTiming));
    c.device = dev;
  }
  *out = c;
  return MOE_OK;
}

moe_status make_tmap_kpair(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           int elem_bytes, uint32_t box_rows) {
  if (elem_bytes != 2 || cols % 128 != 0) return MOE_ERR_UNSUPPORTED;
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (g_encode == nullptr) {
    record_cuda_error_text("cuTensorMapEncodeTiled is unavailable");
    return MOE_ERR_CUDA;
  }
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0) return MOE_ERR_INVALID_ARG;
  // dims (innermost first): 64 elements of a column block, rows, column blocks
  cuuint64_t dims[3] = {64, rows, cols / 64};
  cuuint64_t strides[2] = {cols * (cuuint64_t)elem_bytes, 64 * (cuuint64_t)elem_bytes};
  cuuint32_t box[3] = {64, box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    record_cuda_error_text("cuTensorMapEncodeTiled (3-d) failed");
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status make_tmap_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                        int elem_bytes, uint32_t box_rows, uint32_t box_cols, int swizzle_bytes) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (g_encode == nullptr) {
    record_cuda_error_text("cuTensorMapEncodeTiled is unavailable");
    return MOE_ERR_CUDA;
  }
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || ((cols * elem_bytes) & 15u) != 0)
    return MOE_ERR_INVALID_ARG;
  CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (cuuint64_t)elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                        : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    record_cuda_error_text("cuTensorMapEncodeTiled failed");
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe

extern "C" {

moe_status moe_read_device_status(moe_stream_t stream, int32_t* status) {
  if (status == nullptr) return MOE_ERR_INVALID_ARG;
  moe::DeviceCtx ctx;
  MOE_TRY(moe::device_ctx(&ctx));
  MOE_TRY_CUDA(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  int v = 0;
  MOE_TRY_CUDA(cudaMemcpyFromSymbol(&v, moe::g_kernel_status, sizeof(int)));
  int zero = 0;
  MOE_TRY_CUDA(cudaMemcpyToSymbol(moe::g_kernel_status, &zero, sizeof(int)));
  *status = v;
  return MOE_OK;
}

const char* moe_status_string(int32_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    case MOE_ERR_DEVICE_BOUNDS: return "MOE_ERR_DEVICE_BOUNDS";
    default: return "MOE_ERR_UNKNOWN";
  }
}

const char* moe_last_cuda_error(void) { return moe::g_last_error; }

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

}  // extern "C"
