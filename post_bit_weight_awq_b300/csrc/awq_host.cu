// Host-side launch helpers shared by the kernel translation units: device
// queries and kernel attributes that are looked up once per device instead
// of on every launch (launch paths such as a decode loop call them per layer),
// and the TMA tensor maps of the tensor-core kernels.
#include <mutex>

#include "awq_launch.h"

namespace awq {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices] = {};

struct SmemEntry {
  const void* func;
  int dev;
  int bytes;
};
constexpr int kMaxEntries = 256;
SmemEntry g_smem[kMaxEntries];
int g_nsmem = 0;

}  // namespace

cudaError_t sm_count(int* sms) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_sms[dev] == 0) {
    e = cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      g_sms[dev] = 0;
      return e;
    }
  }
  *sms = g_sms[dev];
  return cudaSuccess;
}

cudaError_t ensure_dynamic_smem(const void* func, int bytes) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < g_nsmem; ++i)
    if (g_smem[i].func == func && g_smem[i].dev == dev) {
      if (g_smem[i].bytes >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e == cudaSuccess) g_smem[i].bytes = bytes;
      return e;
    }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && g_nsmem < kMaxEntries) g_smem[g_nsmem++] = {func, dev, bytes};
  return e;
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once (thread-safe).
EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return (EncodeTiledFn) nullptr;
  }();
  return fn;
}

}  // namespace

bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t strides[2];
  strides[0] = dims[0] * 2;
  if (rank == 3) strides[1] = dims[0] * dims[1] * 2;
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), dims,
                        strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace awq
