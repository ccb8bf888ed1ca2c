// awq_act_stats_noalloc: the activation statistic without caller scratch.
//
// Some callers cannot call cudaMalloc or hand the library a scratch buffer:
// a plugin inside an inference engine or training framework that owns all
// device memory and passes the plugin only its input and output pointers, or
// code on a latency-critical path where a cudaMalloc (which may synchronise
// the device) is not allowed. For them this entry point runs the same kernels
// as awq_act_stats, with the per-chunk partial sums in a fixed-size array of
// this library's own device memory instead of a caller workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (4 MiB + 16 KiB) until the process exits. In host code
// its name is only a host-side stand-in, so its device address is looked up
// with cudaGetSymbolAddress, with the device current, on the first call made
// in each context of a device (the first call on the device, and again
// after a cudaDeviceReset, which reloads the module, possibly elsewhere);
// that first call should come before any stream capture. All calls share the
// array and it keeps the last call's contents; the kernel writes every
// partial it later reads, and each call clears the strips' ticket counters
// (the part that must start at zero) with a memset on its stream before the
// kernel runs. Calls whose work overlaps on the GPU (two streams, or two
// host threads) race on the array: serialise them.
#include <cuda.h>

#include <mutex>

#include "awq.h"
#include "awq_launch.h"
#include "awq_trace.h"

namespace {

constexpr size_t kScratchFloats = AWQ_NOALLOC_STATS_MAX_FLOATS;
// stats_chunks(n_tok, in) * in <= kScratchFloats implies in <= kScratchFloats,
// so at most kScratchFloats / 256 strips of 256 channels need a ticket counter.
constexpr size_t kTicketWords = kScratchFloats / 256;
static __device__ __align__(256) float g_stats_scratch[kScratchFloats + kTicketWords];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchAddress {
  unsigned long long ctx_id = 0;  // context the address belongs to (0: none yet)
  float* ptr = nullptr;
};
ScratchAddress g_scratch[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Identifier of the current context (driver entry points looked up once).
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  if (get_current == nullptr || get_id == nullptr) {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) != cudaSuccess ||
        qa != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
        qb != cudaDriverEntryPointSuccess)
      return false;
    get_current = reinterpret_cast<CtxGetCurrentFn>(a);
    get_id = reinterpret_cast<CtxGetIdFn>(b);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current device's context (set
// up once per context).
awq_status scratch_on_current_device(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return AWQ_ERR_CUDA;
  // makes the device's primary context current (it exists after this call)
  if (cudaSetDevice(dev) != cudaSuccess) return AWQ_ERR_CUDA;
  unsigned long long id = 0;
  if (!current_context_id(&id)) return AWQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchAddress& a = g_scratch[dev];
  if (a.ptr == nullptr || a.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_stats_scratch) != cudaSuccess || p == nullptr) return AWQ_ERR_CUDA;
    a.ptr = static_cast<float*>(p);
    a.ctx_id = id;
  }
  *out = a.ptr;
  return AWQ_OK;
}

}  // namespace

extern "C" awq_status awq_act_stats_noalloc(const void* X, int32_t x_dtype, int64_t n_tok, int64_t in,
                                            float* mean_abs, awq_stream_t stream) {
  AWQ_TRACE("awq_act_stats_noalloc");
  if (X == nullptr || mean_abs == nullptr) return AWQ_ERR_INVALID_ARG;
  if (x_dtype == AWQ_FP32) return AWQ_ERR_UNSUPPORTED;
  if (x_dtype != AWQ_BF16) return AWQ_ERR_INVALID_ARG;
  if (n_tok < 1 || in < 1 || in % 8 != 0 || n_tok > ((int64_t)1 << 30) || in > ((int64_t)1 << 30))
    return AWQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(X) & 15u) || (reinterpret_cast<uintptr_t>(mean_abs) & 15u))
    return AWQ_ERR_MISALIGNED;
  if ((size_t)awq::stats_chunks(n_tok, in) * (size_t)in > kScratchFloats) return AWQ_ERR_WORKSPACE;
  float* scratch = nullptr;
  const awq_status st = scratch_on_current_device(&scratch);
  if (st != AWQ_OK) return st;
  uint32_t* tickets = reinterpret_cast<uint32_t*>(scratch + kScratchFloats);
  const cudaError_t e = awq::launch_stats(static_cast<const uint16_t*>(X), n_tok, in, scratch, tickets, mean_abs,
                                          (cudaStream_t)stream);
  return e == cudaSuccess ? AWQ_OK : AWQ_ERR_CUDA;
}
