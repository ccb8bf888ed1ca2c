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
// min(s_i)). The scale decides the codes, so it is formed in fp64 (pow,
// product, sqrt, quotient) and rounded to fp32 once. Because x^alpha is
// non-decreasing in x for alpha >= 0, max(s_i) and min(s_i) are the powers of
// the largest and smallest clamped statistic; every block finds those two
// with a fixed-order reduction and forms the normaliser itself.
// Grid: (ceil(in / 256), n_grid). alpha = 0 gives s = 1 exactly.

__global__ void __launch_bounds__(256) alpha_scales_kernel(const float* __restrict__ mean_abs, int K, int G,
                                                           double clamp_min, int normalize,
                                                           float* __restrict__ s_out,
                                                           float* __restrict__ inv_out) {
  __shared__ float smax[8], smin[8];
  __shared__ double norm_sh;
  const int i = blockIdx.y;
  const double alpha = (double)i / (double)G;
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
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
      smax[0] = fmaxf(smax[0], smax[w]);
      smin[0] = fminf(smin[0], smin[w]);
    }
    double c = 1.0;
    if (normalize) {
      const double hi = pow(fmax((double)smax[0], clamp_min), alpha);
      const double lo = pow(fmax((double)smin[0], clamp_min), alpha);
      c = sqrt(hi * lo);
    }
    norm_sh = c;
  }
  __syncthreads();
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j < K) {
    const double sj = pow(fmax((double)mean_abs[j], clamp_min), alpha) / norm_sh;
    const float s32 = (float)sj;
    s_out[(size_t)i * K + j] = s32;
    inv_out[(size_t)i * K + j] = __fdiv_rn(1.0f, s32);
  }
}

cudaError_t launch_alpha_scales(const float* mean_abs, int64_t K, const awq_config& cfg, float* s,
                                float* inv_s, cudaStream_t st) {
  dim3 grid((unsigned)((K + 255) / 256), (unsigned)cfg.n_grid);
  alpha_scales_kernel<<<grid, 256, 0, st>>>(mean_abs, (int)K, cfg.n_grid, (double)cfg.sx_clamp_min,
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
// with 8 weights each (one 16-byte load); each lane holds the same 8 columns
// of kRows consecutive rows, so one load of s_i / (1/s_i) serves kRows groups.
// W is read once and every alpha is produced from registers.
// RESIDUAL writes bf16(W_hat_i - W); REFERENCE writes bf16(W_hat_i) and, in
// slot G, bf16(W).

constexpr int kFqRows = 2;

template <typename WT, bool REF>
__global__ void __launch_bounds__(256) fakequant_kernel(const WT* __restrict__ W, int N, int K, int G,
                                                        const float* __restrict__ s,
                                                        const float* __restrict__ inv_s, float qmax,
                                                        float floor_, uint16_t* __restrict__ op,
                                                        int64_t slot_elems, int64_t units) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t unit = t >> 4;  // (row block, column group)
  const int sub = (int)(t & 15);
  const bool valid_unit = unit < units;
  const int cgroups = K >> 7;
  const int64_t u = valid_unit ? unit : 0;
  const int row0 = (int)(u / cgroups) * kFqRows;
  const int col = (int)(u % cgroups) * 128 + sub * 8;
  float w[kFqRows][8];
  bool rv[kFqRows];
#pragma unroll
  for (int i = 0; i < kFqRows; ++i) {
    rv[i] = valid_unit && (row0 + i < N);
    const int r = rv[i] ? row0 + i : 0;
    WLoad<WT>::load8(W + (size_t)r * K + col, w[i]);
    if (REF && rv[i]) {
      uint4 o;
      o.x = pack_bf16x2(w[i][0], w[i][1]);
      o.y = pack_bf16x2(w[i][2], w[i][3]);
      o.z = pack_bf16x2(w[i][4], w[i][5]);
      o.w = pack_bf16x2(w[i][6], w[i][7]);
      *reinterpret_cast<uint4*>(op + (size_t)G * slot_elems + (size_t)r * K + col) = o;
    }
  }
  for (int a = 0; a < G; ++a) {
    float sv[8], iv[8];
    load8f(s + (size_t)a * K + col, sv);
    load8f(inv_s + (size_t)a * K + col, iv);
#pragma unroll
    for (int i = 0; i < kFqRows; ++i) {
      float v[8];
      float mn = INFINITY, mx = -INFINITY;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        v[e] = __fmul_rn(w[i][e], sv[e]);
        mn = fminf(mn, v[e]);
        mx = fmaxf(mx, v[e]);
      }
#pragma unroll
      for (int o = 8; o; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      const GroupFast g = group_fast(mn, mx, qmax, floor_);
      float r8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float qz = quant_code_minus_z(v[e], g);  // q - z
        const float dq = __fmul_rn(qz, g.delta);      // dequantised, scaled space
        r8[e] = REF ? __fmul_rn(dq, iv[e]) : fmaf(dq, iv[e], -w[i][e]);
      }
      if (rv[i]) {
        uint4 o;
        o.x = pack_bf16x2(r8[0], r8[1]);
        o.y = pack_bf16x2(r8[2], r8[3]);
        o.z = pack_bf16x2(r8[4], r8[5]);
        o.w = pack_bf16x2(r8[6], r8[7]);
        *reinterpret_cast<uint4*>(op + (size_t)a * slot_elems + (size_t)(row0 + i) * K + col) = o;
      }
    }
  }
}

cudaError_t launch_fakequant(const void* W, int w_dtype, int64_t N, int64_t K, const float* s,
                             const float* inv_s, const awq_config& cfg, uint16_t* op, cudaStream_t st) {
  const int64_t units = (N + kFqRows - 1) / kFqRows * (K / 128);
  const unsigned blocks = (unsigned)((units * 16 + 255) / 256);
  const float qmax = (float)((1 << cfg.w_bit) - 1);
  const bool ref = cfg.loss_form == AWQ_LOSS_REFERENCE;
  const int64_t slot = N * K;
  const int n = (int)N, k = (int)K, g = cfg.n_grid;
  const float fl = cfg.delta_floor;
  if (w_dtype == AWQ_BF16) {
    if (ref)
      fakequant_kernel<uint16_t, true><<<blocks, 256, 0, st>>>((const uint16_t*)W, n, k, g, s, inv_s, qmax, fl, op,
                                                               slot, units);
    else
      fakequant_kernel<uint16_t, false><<<blocks, 256, 0, st>>>((const uint16_t*)W, n, k, g, s, inv_s, qmax, fl,
                                                                op, slot, units);
  } else {
    if (ref)
      fakequant_kernel<float, true><<<blocks, 256, 0, st>>>((const float*)W, n, k, g, s, inv_s, qmax, fl, op, slot,
                                                            units);
    else
      fakequant_kernel<float, false><<<blocks, 256, 0, st>>>((const float*)W, n, k, g, s, inv_s, qmax, fl, op,
                                                             slot, units);
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
  const GroupFast g = group_fast(mn, mx, qmax, floor_);
  const float z = -g.lo;
  uint32_t words[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t wd = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) wd |= (uint32_t)__fadd_rn(quant_code_minus_z(v[k * 8 + e], g), z) << (4 * e);
    words[k] = wd;
  }
  if (valid) {
    *reinterpret_cast<uint4*>(qweight + gid * 16 + sub * 4) = make_uint4(words[0], words[1], words[2], words[3]);
    if (sub == 0) {
      scales[gid] = __half_as_ushort(__float2half_rn(g.delta));
      zeros[gid] = __half_as_ushort(__float2half_rn(z));
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
