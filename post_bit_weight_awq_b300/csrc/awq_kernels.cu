// Bandwidth-bound kernels of the AWQ per-layer search and pack (sm_103a):
//   stats_partial / stats_finalize : mean |x| per input channel
//   alpha_scales                   : s_i = max(sx, clamp)^alpha_i, normalised
//   fakequant                      : the search operand for every alpha
//   pack                           : final INT4 codes, fp16 scales and zeros
//   loss_select                    : per-alpha loss, first argmin, s_best
#include <math.h>

#include "awq_device.cuh"
#include "awq_launch.h"

namespace awq {

// ============================================================== statistics
//
// mean_t |X[t, j]| ("AWQ: How Activation-Aware Quantization Saves 4-bit
// LLMs", "How does AWQ decide which weights to protect?"; "AWQ > Summary",
// "Salient weight identification").
//
// Block = 32 x 8 threads over a strip of 256 channels and a chunk of
// kStatsRows tokens. Each thread reads 8 channels (16 B) of every 8th row of
// the chunk, so a warp reads 512 contiguous bytes per row. The 8 row phases
// are added in fixed order in shared memory; chunks are added in fp64 by the
// finalize kernel in fixed order. The result is deterministic.

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void acc_abs_bf16x8(float (&a)[8], const uint4& v) {
  a[0] += fabsf(bf16_lo(v.x));
  a[1] += fabsf(bf16_hi(v.x));
  a[2] += fabsf(bf16_lo(v.y));
  a[3] += fabsf(bf16_hi(v.y));
  a[4] += fabsf(bf16_lo(v.z));
  a[5] += fabsf(bf16_hi(v.z));
  a[6] += fabsf(bf16_lo(v.w));
  a[7] += fabsf(bf16_hi(v.w));
}

__global__ void __launch_bounds__(256) stats_partial_kernel(const uint16_t* __restrict__ X, int n, int K,
                                                            float* __restrict__ partials) {
  __shared__ float red[8][256 + 8];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int col = (blockIdx.x * 32 + tx) * 8;
  const int r0 = blockIdx.y * kStatsRows;
  const int r1 = min(r0 + kStatsRows, n);
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (col < K) {
    int r = r0 + ty;
    for (; r + 24 < r1; r += 32) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = ld_nc_v4(X + (size_t)(r + 8 * u) * K + col);
#pragma unroll
      for (int u = 0; u < 4; ++u) acc_abs_bf16x8(a, v[u]);
    }
    for (; r < r1; r += 8) acc_abs_bf16x8(a, ld_nc_v4(X + (size_t)r * K + col));
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) red[ty][tx * 8 + i] = a[i];
  __syncthreads();
  const int t = ty * 32 + tx;
  float sum = 0.f;
#pragma unroll
  for (int y = 0; y < 8; ++y) sum += red[y][t];
  const int c = blockIdx.x * 256 + t;
  if (c < K) partials[(size_t)blockIdx.y * K + c] = sum;
}

__global__ void __launch_bounds__(256) stats_finalize_kernel(const float* __restrict__ partials, int chunks,
                                                             int n, int K, float* __restrict__ mean_abs) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= K) return;
  double s = 0.0;
  for (int i = 0; i < chunks; ++i) s += (double)partials[(size_t)i * K + c];
  mean_abs[c] = (float)(s / (double)n);
}

cudaError_t launch_stats(const uint16_t* X, int64_t n, int64_t K, float* partials, float* mean_abs,
                         cudaStream_t st) {
  const int chunks = stats_chunks(n);
  dim3 grid((unsigned)((K + 255) / 256), (unsigned)chunks);
  stats_partial_kernel<<<grid, dim3(32, 8), 0, st>>>(X, (int)n, (int)K, partials);
  stats_finalize_kernel<<<(unsigned)((K + 255) / 256), 256, 0, st>>>(partials, chunks, (int)n, (int)K,
                                                                      mean_abs);
  return cudaGetLastError();
}

// ============================================================== alpha scales
//
// One block per alpha_i = i / n_grid: s = max(sx, clamp)^alpha ("AWQ: How
// Activation-Aware Quantization Saves 4-bit LLMs", search_scale listing;
// "AWQ > Summary", "The scaling formula"), then optionally s /= sqrt(max(s) *
// min(s)). alpha = 0 gives s = 1 exactly (pow(x, 0) = 1, and sqrt(1*1) = 1).

__global__ void __launch_bounds__(256) alpha_scales_kernel(const float* __restrict__ mean_abs, int K, int G,
                                                           float clamp_min, int normalize,
                                                           float* __restrict__ s_out,
                                                           float* __restrict__ inv_out) {
  __shared__ float smax[8], smin[8];
  const int i = blockIdx.x;
  const float alpha = __fdiv_rn((float)i, (float)G);
  float mx = -INFINITY, mn = INFINITY;
  for (int j = threadIdx.x; j < K; j += blockDim.x) {
    const float sj = powf(fmaxf(mean_abs[j], clamp_min), alpha);
    mx = fmaxf(mx, sj);
    mn = fminf(mn, sj);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    smax[warp] = mx;
    smin[warp] = mn;
  }
  __syncthreads();
  mx = smax[0];
  mn = smin[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
    mx = fmaxf(mx, smax[w]);
    mn = fminf(mn, smin[w]);
  }
  const float c = normalize ? sqrtf(__fmul_rn(mx, mn)) : 1.0f;
  for (int j = threadIdx.x; j < K; j += blockDim.x) {
    const float sj = __fdiv_rn(powf(fmaxf(mean_abs[j], clamp_min), alpha), c);
    s_out[(size_t)i * K + j] = sj;
    inv_out[(size_t)i * K + j] = __fdiv_rn(1.0f, sj);
  }
}

cudaError_t launch_alpha_scales(const float* mean_abs, int64_t K, const awq_config& cfg, float* s,
                                float* inv_s, cudaStream_t st) {
  alpha_scales_kernel<<<cfg.n_grid, 256, 0, st>>>(mean_abs, (int)K, cfg.n_grid, cfg.sx_clamp_min,
                                                  cfg.normalize, s, inv_s);
  return cudaGetLastError();
}

// ============================================================== weight loads

template <typename WT>
struct WLoad;

template <>
struct WLoad<uint16_t> {  // bf16 bits
  static __device__ __forceinline__ void load8(const uint16_t* p, float (&w)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    w[0] = bf16_lo(v.x);
    w[1] = bf16_hi(v.x);
    w[2] = bf16_lo(v.y);
    w[3] = bf16_hi(v.y);
    w[4] = bf16_lo(v.z);
    w[5] = bf16_hi(v.z);
    w[6] = bf16_lo(v.w);
    w[7] = bf16_hi(v.w);
  }
};

template <>
struct WLoad<float> {
  static __device__ __forceinline__ void load8(const float* p, float (&w)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    w[0] = a.x;
    w[1] = a.y;
    w[2] = a.z;
    w[3] = a.w;
    w[4] = b.x;
    w[5] = b.y;
    w[6] = b.z;
    w[7] = b.w;
  }
};

__device__ __forceinline__ void load8f(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x;
  v[1] = a.y;
  v[2] = a.z;
  v[3] = a.w;
  v[4] = b.x;
  v[5] = b.y;
  v[6] = b.z;
  v[7] = b.w;
}

// ============================================================== fake-quant
//
// For every alpha_i: W_hat_i = Q(W * s_i) * (1 / s_i), the scale-quantise-
// fold-back step of the search_scale listing ("AWQ: How Activation-Aware
// Quantization Saves 4-bit LLMs"), justified by the scaling equation of "AWQ
// > Salient Weight Preservation". A group of 128 weights is held by 16 lanes
// (8 weights each, one 16-byte load); W is read once and all alphas are
// produced from registers. RESIDUAL writes bf16(W_hat_i - W); REFERENCE
// writes bf16(W_hat_i) and, in slot G, bf16(W).

template <typename WT, bool REF>
__global__ void __launch_bounds__(256) fakequant_kernel(const WT* __restrict__ W, int64_t ngroups, int K, int G,
                                                        const float* __restrict__ s,
                                                        const float* __restrict__ inv_s, float qmax,
                                                        float floor_, uint16_t* __restrict__ op,
                                                        int64_t slot_elems) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t gid = t >> 4;
  const int sub = (int)(t & 15);
  const bool valid = gid < ngroups;
  const int64_t off = (valid ? gid : 0) * 128 + sub * 8;
  const int col = (int)(off % K);
  float w[8];
  WLoad<WT>::load8(W + off, w);
  if (REF && valid) {
    uint4 o;
    o.x = pack_bf16x2(w[0], w[1]);
    o.y = pack_bf16x2(w[2], w[3]);
    o.z = pack_bf16x2(w[4], w[5]);
    o.w = pack_bf16x2(w[6], w[7]);
    *reinterpret_cast<uint4*>(op + (size_t)G * slot_elems + off) = o;
  }
  for (int a = 0; a < G; ++a) {
    float sv[8], iv[8], v[8];
    load8f(s + (size_t)a * K + col, sv);
    load8f(inv_s + (size_t)a * K + col, iv);
    float mn = INFINITY, mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      v[e] = __fmul_rn(w[e], sv[e]);
      mn = fminf(mn, v[e]);
      mx = fmaxf(mx, v[e]);
    }
#pragma unroll
    for (int o = 8; o; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const GroupQ g = group_params(mn, mx, qmax, floor_);
    float r[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float q = quant_code(v[e], g, qmax);
      const float wh = __fmul_rn(__fmul_rn(__fsub_rn(q, g.z), g.delta), iv[e]);
      r[e] = REF ? wh : __fsub_rn(wh, w[e]);
    }
    if (valid) {
      uint4 o;
      o.x = pack_bf16x2(r[0], r[1]);
      o.y = pack_bf16x2(r[2], r[3]);
      o.z = pack_bf16x2(r[4], r[5]);
      o.w = pack_bf16x2(r[6], r[7]);
      *reinterpret_cast<uint4*>(op + (size_t)a * slot_elems + off) = o;
    }
  }
}

cudaError_t launch_fakequant(const void* W, int w_dtype, int64_t N, int64_t K, const float* s,
                             const float* inv_s, const awq_config& cfg, uint16_t* op, cudaStream_t st) {
  const int64_t ngroups = N * K / 128;
  const int64_t threads = ngroups * 16;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  const float qmax = (float)((1 << cfg.w_bit) - 1);
  const bool ref = cfg.loss_form == AWQ_LOSS_REFERENCE;
  const int64_t slot = N * K;
  if (w_dtype == AWQ_BF16) {
    if (ref)
      fakequant_kernel<uint16_t, true><<<blocks, 256, 0, st>>>((const uint16_t*)W, ngroups, (int)K, cfg.n_grid,
                                                               s, inv_s, qmax, cfg.delta_floor, op, slot);
    else
      fakequant_kernel<uint16_t, false><<<blocks, 256, 0, st>>>((const uint16_t*)W, ngroups, (int)K,
                                                                cfg.n_grid, s, inv_s, qmax, cfg.delta_floor, op,
                                                                slot);
  } else {
    if (ref)
      fakequant_kernel<float, true><<<blocks, 256, 0, st>>>((const float*)W, ngroups, (int)K, cfg.n_grid, s,
                                                            inv_s, qmax, cfg.delta_floor, op, slot);
    else
      fakequant_kernel<float, false><<<blocks, 256, 0, st>>>((const float*)W, ngroups, (int)K, cfg.n_grid, s,
                                                             inv_s, qmax, cfg.delta_floor, op, slot);
  }
  return cudaGetLastError();
}

// ============================================================== pack
//
// Final codes of W * diag(s) with the same quantiser, 8 codes per int32
// ("What is AWQ Quantization? ...", "INT4 Weight Packing & Export"), one fp16
// scale ("AWQ (Activation-Aware Weight Quantization) - AI Glossary", memory
// example) and one fp16 zero per group. A group is held by 4 lanes with 32
// weights each; every lane writes its 4 words with one 128-bit store.

template <typename WT>
__global__ void __launch_bounds__(256) pack_kernel(const WT* __restrict__ W, int64_t ngroups, int K,
                                                   const float* __restrict__ s, float qmax, float floor_,
                                                   int32_t* __restrict__ qweight, uint16_t* __restrict__ scales,
                                                   uint16_t* __restrict__ zeros) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t gid = t >> 2;
  const int sub = (int)(t & 3);
  const bool valid = gid < ngroups;
  const int64_t off = (valid ? gid : 0) * 128 + sub * 32;
  const int col = (int)(off % K);
  float v[32];
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float w[8], sv[8];
    WLoad<WT>::load8(W + off + c * 8, w);
    load8f(s + col + c * 8, sv);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      v[c * 8 + e] = __fmul_rn(w[e], sv[e]);
      mn = fminf(mn, v[c * 8 + e]);
      mx = fmaxf(mx, v[c * 8 + e]);
    }
  }
#pragma unroll
  for (int o = 2; o; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const GroupQ g = group_params(mn, mx, qmax, floor_);
  uint32_t words[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t wd = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) wd |= (uint32_t)quant_code(v[k * 8 + e], g, qmax) << (4 * e);
    words[k] = wd;
  }
  if (valid) {
    *reinterpret_cast<uint4*>(qweight + gid * 16 + sub * 4) = make_uint4(words[0], words[1], words[2], words[3]);
    if (sub == 0) {
      scales[gid] = __half_as_ushort(__float2half_rn(g.delta));
      zeros[gid] = __half_as_ushort(__float2half_rn(g.z));
    }
  }
}

cudaError_t launch_pack(const void* W, int w_dtype, int64_t N, int64_t K, const float* s, const awq_config& cfg,
                        int32_t* qweight, uint16_t* scales, uint16_t* zeros, cudaStream_t st) {
  const int64_t ngroups = N * K / 128;
  const unsigned blocks = (unsigned)((ngroups * 4 + 255) / 256);
  const float qmax = (float)((1 << cfg.w_bit) - 1);
  if (w_dtype == AWQ_BF16)
    pack_kernel<uint16_t><<<blocks, 256, 0, st>>>((const uint16_t*)W, ngroups, (int)K, s, qmax, cfg.delta_floor,
                                                  qweight, scales, zeros);
  else
    pack_kernel<float><<<blocks, 256, 0, st>>>((const float*)W, ngroups, (int)K, s, qmax, cfg.delta_floor,
                                               qweight, scales, zeros);
  return cudaGetLastError();
}

// ============================================================== loss + argmin
//
// L_i = (sum of the tile partials of alpha_i) / (n_tok * out), summed in
// fp64 in a fixed order; the first strict minimum wins ("AWQ: How
// Activation-Aware Quantization Saves 4-bit LLMs", search_scale listing:
// keep an alpha only if its error is strictly lower). One block.

__global__ void __launch_bounds__(1024) loss_select_kernel(const float* __restrict__ partials, int G,
                                                           int64_t per_alpha, double denom,
                                                           const float* __restrict__ s, int K,
                                                           float* __restrict__ losses, int32_t* __restrict__ best_idx,
                                                           float* __restrict__ s_best, uint32_t* status) {
  __shared__ double wsum[32];
  __shared__ double sums[kMaxGrid];
  __shared__ int best_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  for (int a = 0; a < G; ++a) {
    double acc = 0.0;
    const float* p = partials + (size_t)a * per_alpha;
    for (int64_t t = threadIdx.x; t < per_alpha; t += blockDim.x) acc += (double)p[t];
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) wsum[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
      double tot = 0.0;
      for (int w = 0; w < nwarps; ++w) tot += wsum[w];
      sums[a] = tot;
      losses[a] = (float)(tot / denom);
      if (!isfinite(tot)) set_status(status, AWQ_ERR_NONFINITE);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    int b = -1;
    double bv = INFINITY;
    for (int a = 0; a < G; ++a)
      if (sums[a] < bv) {
        bv = sums[a];
        b = a;
      }
    if (b < 0) b = 0;
    best_sh = b;
    *best_idx = b;
  }
  __syncthreads();
  const int b = best_sh;
  for (int j = threadIdx.x; j < K; j += blockDim.x) s_best[j] = s[(size_t)b * K + j];
}

cudaError_t launch_loss_select(const float* partials, int G, int64_t per_alpha, int64_t n_tok, int64_t N,
                               const float* s, int64_t K, float* losses, int32_t* best_idx, float* s_best,
                               uint32_t* status, cudaStream_t st) {
  loss_select_kernel<<<1, 1024, 0, st>>>(partials, G, per_alpha, (double)n_tok * (double)N, s, (int)K, losses,
                                         best_idx, s_best, status);
  return cudaGetLastError();
}

}  // namespace awq
