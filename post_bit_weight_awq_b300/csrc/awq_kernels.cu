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
// are added in fixed order in shared memory; the finalize kernel adds the
// chunks with a compensated fp32 sum in fixed order. Deterministic.

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
  // compensated (Neumaier) fp32 sum over the chunks, fixed order
  float sum = 0.0f, comp = 0.0f;
  for (int i = 0; i < chunks; ++i) {
    const float x = partials[(size_t)i * K + c];
    const float t = __fadd_rn(sum, x);
    comp = __fadd_rn(comp, fabsf(sum) >= fabsf(x) ? __fadd_rn(__fsub_rn(sum, t), x) : __fadd_rn(__fsub_rn(x, t), sum));
    sum = t;
  }
  mean_abs[c] = (float)(((double)sum + (double)comp) / (double)n);
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
// s_i = max(sx, clamp)^alpha_i ("AWQ: How Activation-Aware Quantization
// Saves 4-bit LLMs", search_scale listing; "AWQ > Summary", "The scaling
// formula"), alpha_i = i / n_grid, then optionally s_i /= sqrt(max(s_i) *
// min(s_i)). The scale decides the codes, so it is formed in fp64 and rounded
// to fp32 once. Since alpha_i = i / n_grid, b^alpha_i = (b^(1/n_grid))^i: one
// pow per channel, then one fp64 product per alpha (the products drift from
// a direct pow by at most ~n_grid fp64 ulps, which changes the fp32-rounded
// scale only when it lies that close to an fp32 rounding boundary). x^alpha
// is non-decreasing in x, so max(s_i) and min(s_i) are the powers of the
// largest and smallest clamped statistic; each block finds those two with a
// fixed-order reduction and forms 1 / sqrt(max * min) per alpha.
// One thread per channel; alpha = 0 gives s = 1 exactly.

__global__ void __launch_bounds__(128) alpha_scales_kernel(const float* __restrict__ mean_abs, int K, int G,
                                                           double clamp_min, int normalize,
                                                           float* __restrict__ s_out,
                                                           float* __restrict__ inv_out) {
  __shared__ float smax[4], smin[4];
  __shared__ double inv_norm[kMaxGrid];
  float mx = -INFINITY, mn = INFINITY;
  for (int j = threadIdx.x; j < K; j += blockDim.x) {
    const float v = mean_abs[j];
    mx = fmaxf(mx, v);
    mn = fminf(mn, v);
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
  if ((int)threadIdx.x < G) {
    const int i = threadIdx.x;
    double c = 1.0;
    if (normalize) {
      float bmx = smax[0], bmn = smin[0];
      for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
        bmx = fmaxf(bmx, smax[w]);
        bmn = fminf(bmn, smin[w]);
      }
      const double alpha = (double)i / (double)G;
      c = sqrt(pow(fmax((double)bmx, clamp_min), alpha) * pow(fmax((double)bmn, clamp_min), alpha));
    }
    inv_norm[i] = 1.0 / c;
  }
  __syncthreads();
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= K) return;
  const double b = fmax((double)mean_abs[j], clamp_min);
  const double root = pow(b, 1.0 / (double)G);
  double p = 1.0;  // b^(i/G)
  for (int i = 0; i < G; ++i) {
    const float s32 = (float)(p * inv_norm[i]);
    s_out[(size_t)i * K + j] = s32;
    inv_out[(size_t)i * K + j] = __fdiv_rn(1.0f, s32);
    p *= root;
  }
}

cudaError_t launch_alpha_scales(const float* mean_abs, int64_t K, const awq_config& cfg, float* s,
                                float* inv_s, cudaStream_t st) {
  alpha_scales_kernel<<<(unsigned)((K + 127) / 128), 128, 0, st>>>(mean_abs, (int)K, cfg.n_grid,
                                                                   (double)cfg.sx_clamp_min, cfg.normalize, s, inv_s);
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

template <typename WT>
__device__ __forceinline__ void load16w(const WT* p, float (&w)[16]) {
  float a[8], b[8];
  WLoad<WT>::load8(p, a);
  WLoad<WT>::load8(p + 8, b);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    w[e] = a[e];
    w[8 + e] = b[e];
  }
}

__device__ __forceinline__ void load16f(const float* p, float (&v)[16]) {
  float a[8], b[8];
  load8f(p, a);
  load8f(p + 8, b);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    v[e] = a[e];
    v[8 + e] = b[e];
  }
}

// Group min/max of 16 values per lane over the 8 lanes of a group.
__device__ __forceinline__ void group_minmax16(const float (&v)[16], float& mn, float& mx) {
  mn = v[0];
  mx = v[0];
#pragma unroll
  for (int e = 1; e < 16; ++e) {
    mn = fminf(mn, v[e]);
    mx = fmaxf(mx, v[e]);
  }
#pragma unroll
  for (int o = 4; o; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
}

// ============================================================== fake-quant
//
// For every alpha_i: W_hat_i = Q(W * s_i) * (1 / s_i), the scale-quantise-
// fold-back step of the search_scale listing ("AWQ: How Activation-Aware
// Quantization Saves 4-bit LLMs"), justified by the scaling equation of "AWQ
// > Salient Weight Preservation". A group of 128 weights is held by 8 lanes
// with 16 weights each (two 16-byte loads); W is read once and every alpha is
// produced from registers, so per alpha a lane does two shuffle steps of the
// group reduction, the group's step, zero point and clamp decision, and 16
// division-free exact code decisions.
// RESIDUAL writes bf16(W_hat_i - W); REFERENCE writes bf16(W_hat_i) and, in
// slot G, bf16(W).

template <typename WT, bool REF>
__global__ void __launch_bounds__(256) fakequant_kernel(const WT* __restrict__ W, int64_t ngroups, int K, int G,
                                                        const float* __restrict__ s,
                                                        const float* __restrict__ inv_s, float qmax,
                                                        float floor_, uint16_t* __restrict__ op,
                                                        int64_t slot_elems) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t gid = t >> 3;
  const int sub = (int)(t & 7);
  const bool valid = gid < ngroups;
  const int64_t off = (valid ? gid : 0) * 128 + sub * 16;
  const int col = (int)(off % K);
  float w[16];
  load16w<WT>(W + off, w);
  if (REF && valid) {
    uint4 o0, o1;
    o0.x = pack_bf16x2(w[0], w[1]);
    o0.y = pack_bf16x2(w[2], w[3]);
    o0.z = pack_bf16x2(w[4], w[5]);
    o0.w = pack_bf16x2(w[6], w[7]);
    o1.x = pack_bf16x2(w[8], w[9]);
    o1.y = pack_bf16x2(w[10], w[11]);
    o1.z = pack_bf16x2(w[12], w[13]);
    o1.w = pack_bf16x2(w[14], w[15]);
    uint4* dst = reinterpret_cast<uint4*>(op + (size_t)G * slot_elems + off);
    dst[0] = o0;
    dst[1] = o1;
  }
  for (int a = 0; a < G; ++a) {
    float v[16], sv[16];
    load16f(s + (size_t)a * K + col, sv);
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __fmul_rn(w[e], sv[e]);
    float mn, mx;
    group_minmax16(v, mn, mx);
    const GroupFast g = group_fast(mn, mx, qmax, floor_);
    float k[16];
    quant_codes_minus_z<16>(v, g, k);  // q - z
    float iv[16];
    load16f(inv_s + (size_t)a * K + col, iv);
    float r[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float dq = __fmul_rn(k[e], g.delta);  // dequantised, scaled space
      r[e] = REF ? __fmul_rn(dq, iv[e]) : fmaf(dq, iv[e], -w[e]);
    }
    if (valid) {
      uint4 o0, o1;
      o0.x = pack_bf16x2(r[0], r[1]);
      o0.y = pack_bf16x2(r[2], r[3]);
      o0.z = pack_bf16x2(r[4], r[5]);
      o0.w = pack_bf16x2(r[6], r[7]);
      o1.x = pack_bf16x2(r[8], r[9]);
      o1.y = pack_bf16x2(r[10], r[11]);
      o1.z = pack_bf16x2(r[12], r[13]);
      o1.w = pack_bf16x2(r[14], r[15]);
      uint4* dst = reinterpret_cast<uint4*>(op + (size_t)a * slot_elems + off);
      dst[0] = o0;
      dst[1] = o1;
    }
  }
}

cudaError_t launch_fakequant(const void* W, int w_dtype, int64_t N, int64_t K, const float* s,
                             const float* inv_s, const awq_config& cfg, uint16_t* op, cudaStream_t st) {
  const int64_t ngroups = N * K / 128;
  const unsigned blocks = (unsigned)((ngroups * 8 + 255) / 256);
  const float qmax = (float)((1 << cfg.w_bit) - 1);
  const bool ref = cfg.loss_form == AWQ_LOSS_REFERENCE;
  const int64_t slot = N * K;
  const int k = (int)K, g = cfg.n_grid;
  const float fl = cfg.delta_floor;
  if (w_dtype == AWQ_BF16) {
    if (ref)
      fakequant_kernel<uint16_t, true><<<blocks, 256, 0, st>>>((const uint16_t*)W, ngroups, k, g, s, inv_s, qmax,
                                                               fl, op, slot);
    else
      fakequant_kernel<uint16_t, false><<<blocks, 256, 0, st>>>((const uint16_t*)W, ngroups, k, g, s, inv_s, qmax,
                                                                fl, op, slot);
  } else {
    if (ref)
      fakequant_kernel<float, true><<<blocks, 256, 0, st>>>((const float*)W, ngroups, k, g, s, inv_s, qmax, fl,
                                                            op, slot);
    else
      fakequant_kernel<float, false><<<blocks, 256, 0, st>>>((const float*)W, ngroups, k, g, s, inv_s, qmax, fl,
                                                             op, slot);
  }
  return cudaGetLastError();
}

// ============================================================== pack
//
// Final codes of W * diag(s) with the same quantiser, 8 codes per int32
// ("What is AWQ Quantization? ...", "INT4 Weight Packing & Export"), one fp16
// scale ("AWQ (Activation-Aware Weight Quantization) - AI Glossary", memory
// example) and one fp16 zero per group. A group is held by 8 lanes with 16
// weights (two words) each; even lanes collect their neighbour's two words
// and write four words with one 128-bit store.

template <typename WT>
__global__ void __launch_bounds__(256) pack_kernel(const WT* __restrict__ W, int64_t ngroups, int K,
                                                   const float* __restrict__ s, float qmax, float floor_,
                                                   int32_t* __restrict__ qweight, uint16_t* __restrict__ scales,
                                                   uint16_t* __restrict__ zeros) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t gid = t >> 3;
  const int sub = (int)(t & 7);
  const bool valid = gid < ngroups;
  const int64_t off = (valid ? gid : 0) * 128 + sub * 16;
  const int col = (int)(off % K);
  float v[16], sv[16];
  load16w<WT>(W + off, v);
  load16f(s + col, sv);
#pragma unroll
  for (int e = 0; e < 16; ++e) v[e] = __fmul_rn(v[e], sv[e]);
  float mn, mx;
  group_minmax16(v, mn, mx);
  const GroupFast g = group_fast(mn, mx, qmax, floor_);
  const float z = -g.lo;
  float k[16];
  quant_codes_minus_z<16>(v, g, k);
  uint32_t w0 = 0, w1 = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    w0 |= (uint32_t)__fadd_rn(k[e], z) << (4 * e);
    w1 |= (uint32_t)__fadd_rn(k[8 + e], z) << (4 * e);
  }
  const uint32_t w2 = __shfl_down_sync(0xffffffffu, w0, 1);
  const uint32_t w3 = __shfl_down_sync(0xffffffffu, w1, 1);
  if (valid) {
    if ((sub & 1) == 0)
      *reinterpret_cast<uint4*>(qweight + gid * 16 + sub * 2) = make_uint4(w0, w1, w2, w3);
    if (sub == 0) {
      scales[gid] = __half_as_ushort(__float2half_rn(g.delta));
      zeros[gid] = __half_as_ushort(__float2half_rn(z));
    }
  }
}

cudaError_t launch_pack(const void* W, int w_dtype, int64_t N, int64_t K, const float* s, const awq_config& cfg,
                        int32_t* qweight, uint16_t* scales, uint16_t* zeros, cudaStream_t st) {
  const int64_t ngroups = N * K / 128;
  const unsigned blocks = (unsigned)((ngroups * 8 + 255) / 256);
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
// L_i = (sum of the tile partials of alpha_i) / (n_tok * out); the first
// strict minimum wins ("AWQ: How Activation-Aware Quantization Saves 4-bit
// LLMs", search_scale listing: an alpha replaces the best only if its error
// is strictly lower). One block per alpha sums its partials (fp32 per
// thread over a fixed stride, fp64 across threads in a fixed tree), then one
// small grid picks the argmin and copies s of that alpha to s_best.

__global__ void __launch_bounds__(256) loss_reduce_kernel(const float* __restrict__ partials, int64_t per_alpha,
                                                          double denom, float* __restrict__ losses,
                                                          uint32_t* status) {
  __shared__ double wsum[8];
  const int a = blockIdx.x;
  const float* p = partials + (size_t)a * per_alpha;
  float acc = 0.0f;
  for (int64_t t = threadIdx.x; t < per_alpha; t += blockDim.x) acc += p[t];
  double d = (double)acc;
#pragma unroll
  for (int o = 16; o; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) wsum[warp] = d;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += wsum[w];
    losses[a] = (float)(tot / denom);
    if (!isfinite(tot)) set_status(status, AWQ_ERR_NONFINITE);
  }
}

__global__ void __launch_bounds__(256) select_kernel(const float* __restrict__ losses, int G,
                                                     const float* __restrict__ s, int K,
                                                     int32_t* __restrict__ best_idx, float* __restrict__ s_best) {
  __shared__ int best_sh;
  if (threadIdx.x == 0) {
    int b = -1;
    float bv = INFINITY;
    for (int a = 0; a < G; ++a) {
      const float v = losses[a];
      if (v < bv) {
        bv = v;
        b = a;
      }
    }
    if (b < 0) b = 0;  // every loss non-finite: the status word says so
    best_sh = b;
    if (blockIdx.x == 0) *best_idx = b;
  }
  __syncthreads();
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j < K) s_best[j] = s[(size_t)best_sh * K + j];
}

cudaError_t launch_loss_select(const float* partials, int G, int64_t per_alpha, int64_t n_tok, int64_t N,
                               const float* s, int64_t K, float* losses, int32_t* best_idx, float* s_best,
                               uint32_t* status, cudaStream_t st) {
  loss_reduce_kernel<<<G, 256, 0, st>>>(partials, per_alpha, (double)n_tok * (double)N, losses, status);
  select_kernel<<<(unsigned)((K + 255) / 256), 256, 0, st>>>(losses, G, s, (int)K, best_idx, s_best);
  return cudaGetLastError();
}

}  // namespace awq
