// Host-side launch helpers shared by the kernel translation units: device
// queries and kernel attributes that are looked up once per device instead
// of on every launch (launch paths such as a decode loop call them per layer).
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

}  // namespace awq
