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
// once per device with cudaGetSymbolAddress, with that device current, on
// the first call made on that device; that first call should come before
// any stream capture. All calls share the array and it keeps the last
// call's contents; the kernel writes every partial it later reads, and each
// call clears the strips' ticket counters (the part that must start at
// zero) with a memset on its stream before the kernel runs. Calls whose work
// overlaps on the GPU (two streams, or two host threads) race on the array:
// serialise them.
#include <mutex>

#include "awq.h"
#include "awq_launch.h"
#include "awq_trace.h"

namespace {

constexpr size_t kScratchFloats = AWQ_NOALLOC_STATS_MAX_FLOATS;
// ceil(n_tok/128) * in <= kScratchFloats implies in <= kScratchFloats, so at
// most kScratchFloats / 256 strips of 256 channels need a ticket counter.
constexpr size_t kTicketWords = kScratchFloats / 256;
static __device__ __align__(256) float g_stats_scratch[kScratchFloats + kTicketWords];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once).
awq_status scratch_on_current_device(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return AWQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_stats_scratch) != cudaSuccess || p == nullptr) return AWQ_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
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
  if ((size_t)awq::stats_chunks(n_tok) * (size_t)in > kScratchFloats) return AWQ_ERR_WORKSPACE;
  float* scratch = nullptr;
  const awq_status st = scratch_on_current_device(&scratch);
  if (st != AWQ_OK) return st;
  uint32_t* tickets = reinterpret_cast<uint32_t*>(scratch + kScratchFloats);
  const cudaError_t e = awq::launch_stats(static_cast<const uint16_t*>(X), n_tok, in, scratch, tickets, mean_abs,
                                          (cudaStream_t)stream);
  return e == cudaSuccess ? AWQ_OK : AWQ_ERR_CUDA;
}
