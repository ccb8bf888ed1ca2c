// Bandwidth- and latency-bound kernels of the AWQ per-layer search and pack
// (sm_103a):
//   stats        : mean |x| per input channel (chunk partials, last block adds)
//   alpha_scales : s_i = max(sx, clamp)^alpha_i, normalised
//   fakequant    : the search operand for every alpha
//   pack         : final INT4 codes, fp16 scales and zeros
//   row_losses   : each output row's share of the loss, from the search's sums
//   loss_select  : per-alpha loss, first argmin, s_best
#include <math.h>

#include "awq_device.cuh"
#include "awq_launch.h"
#include "awq_quant.cuh"

namespace awq {

// ============================================================== statistics
//
// mean_t |X[t, j]| ("AWQ: How Activation-Aware Quantization Saves 4-bit
// LLMs", "How does AWQ decide which weights to protect?"; "AWQ > Summary",
// "Salient weight identification").
//
// One launch, one wave. Block = 32 x 8 threads over a strip of 256 channels
// and a chunk of tokens (stats_chunk_rows: about kStatsTargetBlocks blocks
// in all, so every block streams a long run of rows instead of the grid
// running many short waves). Each thread reads 8 channels (16 B) of every
// 8th row of the chunk, so a warp reads 512 contiguous bytes per row; loads
// go in batches of 4 rows, the next batch issued before the current one is
// added, so 4 to 8 loads per thread stay in flight. The 8 row phases are
// added in fixed order in shared memory and the chunk's partial sums go to
// scratch. The block that finishes last on a strip (a ticket counter per
// strip, zeroed before the launch) adds that strip's chunks with a
// compensated fp32 sum in chunk order and writes the mean: the result does
// not depend on which block finishes last, and the chunking depends only on
// the shape. Deterministic.

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

constexpr int kStatsBatch = 4;  // rows per load batch of a thread

// Rows r, r + 8, r + 16, r + 24 of the thread's phase (zeros past the chunk).
__device__ __forceinline__ void stats_load_batch(const uint16_t* __restrict__ X, int r, int r1, int K, int col,
                                                 size_t total, uint4 (&v)[kStatsBatch]) {
#pragma unroll
  for (int u = 0; u < kStatsBatch; ++u) {
    const int row = r + 8 * u;
    const size_t off = (size_t)row * K + col;
    v[u] = row < r1 && AWQ_IN(off, 8, total) ? ld_nc_v4(X + off) : make_uint4(0u, 0u, 0u, 0u);
  }
}

__global__ void __launch_bounds__(256, 4) stats_kernel(const uint16_t* __restrict__ X, int n, int K, int chunk_rows,
                                                    float* __restrict__ partials, uint32_t* __restrict__ tickets,
                                                    float* __restrict__ mean_abs) {
  __shared__ float red[8][256 + 8];
  __shared__ bool last;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int col = (blockIdx.x * 32 + tx) * 8;
  const int r0 = blockIdx.y * chunk_rows;
  const int r1 = min(r0 + chunk_rows, n);
  const size_t total = (size_t)n * K;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (col < K) {
    uint4 cur[kStatsBatch], nxt[kStatsBatch];
    int r = r0 + ty;
    stats_load_batch(X, r, r1, K, col, total, cur);
    for (; r < r1; r += 8 * kStatsBatch) {
      stats_load_batch(X, r + 8 * kStatsBatch, r1, K, col, total, nxt);
#pragma unroll
      for (int u = 0; u < kStatsBatch; ++u) acc_abs_bf16x8(a, cur[u]);
#pragma unroll
      for (int u = 0; u < kStatsBatch; ++u) cur[u] = nxt[u];
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) red[ty][tx * 8 + i] = a[i];
  __syncthreads();
  const int t = ty * 32 + tx;
  float sum = 0.f;
#pragma unroll
  for (int y = 0; y < 8; ++y) sum += red[y][t];
  const int c = blockIdx.x * 256 + t;
  if (c < K && AWQ_IN((size_t)blockIdx.y * K + c, 1, (size_t)gridDim.y * K)) partials[(size_t)blockIdx.y * K + c] = sum;
  // publish this chunk, then find out whether it was the strip's last one
  __threadfence();
  __syncthreads();
  if (t == 0) last = atomicAdd(&tickets[blockIdx.x], 1u) == gridDim.y - 1;
  __syncthreads();
  if (!last || c >= K) return;
  __threadfence();
  // compensated (Neumaier) fp32 sum over the chunks, fixed order; the other
  // blocks' partials are read past L1, 32 chunks' loads in flight at a time
  const int chunks = (int)gridDim.y;
  float s = 0.0f, comp = 0.0f;
  for (int i0 = 0; i0 < chunks; i0 += 32) {
    float xb[32];
#pragma unroll
    for (int u = 0; u < 32; ++u)
      xb[u] = i0 + u < chunks && AWQ_IN((size_t)(i0 + u) * K + c, 1, (size_t)chunks * K)
                  ? __ldcg(partials + (size_t)(i0 + u) * K + c)
                  : 0.0f;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      if (i0 + u >= chunks) break;
      const float x = xb[u];
      const float v = __fadd_rn(s, x);
      comp = __fadd_rn(comp, fabsf(s) >= fabsf(x) ? __fadd_rn(__fsub_rn(s, v), x) : __fadd_rn(__fsub_rn(x, v), s));
      s = v;
    }
  }
  if (AWQ_IN(c, 1, K)) mean_abs[c] = (float)(((double)s + (double)comp) / (double)n);
}

cudaError_t launch_stats(const uint16_t* X, int64_t n, int64_t K, float* partials, uint32_t* tickets,
                         float* mean_abs, cudaStream_t st) {
  const int chunks = stats_chunks(n, K);
  const unsigned strips = (unsigned)stats_strips(K);
  cudaError_t e = cudaMemsetAsync(tickets, 0, strips * sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  stats_kernel<<<dim3(strips, (unsigned)chunks), dim3(32, 8), 0, st>>>(X, (int)n, (int)K, (int)stats_chunk_rows(n, K),
                                                                       partials, tickets, mean_abs);
  return cudaGetLastError();
}

// ============================================================== alpha scales
//
// s_i = max(sx, clamp)^alpha_i ("AWQ: How Activation-Aware Quantization
// Saves 4-bit LLMs", search_scale listing; "AWQ > Summary", "The scaling
// formula"), alpha_i = i / n_grid, then optionally s_i /= sqrt(max(s_i) *
// min(s_i)). The scale decides the codes, so it is formed in fp64 and rounded
// to fp32 once. x^alpha is non-decreasing in x, so max(s_i) and min(s_i) are
// the powers of the largest and smallest clamped statistic, hi and lo, and
//   s_i = b^(i/G) / (hi^(i/G) lo^(i/G))^(1/2) = (b / sqrt(hi lo))^(i/G):
// one fp64 pow per channel gives the root r = (b / sqrt(hi lo))^(1/G), and
// s_i = r^i follows by fp64 products (they drift from a direct pow by at most
// ~n_grid fp64 ulps, which changes the fp32-rounded scale only when it lies
// that close to an fp32 rounding boundary). alpha = 0 gives s = 1 exactly.
// fp64 runs at 1/64 of the fp32 rate on this GPU, so the kernel is a chain of
// latencies kept short: 64 channels per block of 256 threads. All threads
// find the statistic's max/min (16-byte loads, one round of them for
// in <= 4096, fixed-order reduction); the first two warps form the 64
// channels' roots (one pow each); then a quad of threads per channel, thread
// p of the quad writing the alphas i = p (mod 4), stepping by root^4.

constexpr int kAlphaChannels = 64;
constexpr int kAlphaThreads = 4 * kAlphaChannels;

__global__ void __launch_bounds__(kAlphaThreads) alpha_scales_kernel(const float* __restrict__ mean_abs, int K,
                                                                     int G, double clamp_min, int normalize,
                                                                     float* __restrict__ s_out,
                                                                     float* __restrict__ inv_out) {
  __shared__ float smax[kAlphaThreads / 32], smin[kAlphaThreads / 32];
  const int phase = threadIdx.x & 3;
  const int j = blockIdx.x * kAlphaChannels + (threadIdx.x >> 2);
  if (normalize) {
    float mx = -INFINITY, mn = INFINITY;
    const float4* m4 = reinterpret_cast<const float4*>(mean_abs);
    const int K4 = K >> 2;  // K is a multiple of 128
#pragma unroll 4
    for (int q = threadIdx.x; q < K4; q += kAlphaThreads) {
      const float4 v = AWQ_IN(4 * (size_t)q, 4, K) ? m4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
      mx = fmax3f(mx, fmaxf(v.x, v.y), fmaxf(v.z, v.w));
      mn = fmin3f(mn, fminf(v.x, v.y), fminf(v.z, v.w));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    if ((threadIdx.x & 31) == 0) {
      smax[threadIdx.x >> 5] = mx;
      smin[threadIdx.x >> 5] = mn;
    }
    __syncthreads();
  }
  // the first two warps form the block's 64 roots with every lane active (an
  // fp64 instruction costs a warp the same whatever its active lanes)
  __shared__ double root_sh[kAlphaChannels];
  if (threadIdx.x < kAlphaChannels) {
    const int jc = blockIdx.x * kAlphaChannels + threadIdx.x;
    double base = fmax(jc < K && AWQ_IN(jc, 1, K) ? (double)mean_abs[jc] : 1.0, clamp_min);
    if (normalize) {
      float hi32 = smax[0], lo32 = smin[0];
#pragma unroll
      for (int w = 1; w < kAlphaThreads / 32; ++w) {
        hi32 = fmaxf(hi32, smax[w]);
        lo32 = fminf(lo32, smin[w]);
      }
      base /= sqrt(fmax((double)hi32, clamp_min) * fmax((double)lo32, clamp_min));
    }
    root_sh[threadIdx.x] = pow(base, 1.0 / (double)G);
  }
  __syncthreads();
  const double root = root_sh[threadIdx.x >> 2];
  if (j >= K) return;
  const double r2 = root * root, step = r2 * r2;
  double p = phase == 0 ? 1.0 : (phase == 1 ? root : (phase == 2 ? r2 : r2 * root));  // root^phase
  for (int i = phase; i < G; i += 4) {
    if (AWQ_IN((size_t)i * K + j, 1, (size_t)G * K)) {
      const float s32 = (float)p;
      s_out[(size_t)i * K + j] = s32;
      inv_out[(size_t)i * K + j] = __fdiv_rn(1.0f, s32);
    }
    p *= step;
  }
}

cudaError_t launch_alpha_scales(const float* mean_abs, int64_t K, const awq_config& cfg, float* s,
                                float* inv_s, cudaStream_t st) {
  alpha_scales_kernel<<<(unsigned)((K + kAlphaChannels - 1) / kAlphaChannels), kAlphaThreads, 0, st>>>(
      mean_abs, (int)K, cfg.n_grid, (double)cfg.sx_clamp_min, cfg.normalize, s, inv_s);
  return cudaGetLastError();
}

// ============================================================== loads

__device__ __forceinline__ void load8f(const float* p, float* v) {
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
// > Salient Weight Preservation".
// RESIDUAL writes bf16(W_hat_i - W); REFERENCE writes bf16(W_hat_i) and, in
// slot G, bf16(W).
//
// A block owns a strip of 512 input channels (four 128-channel blocks) and a
// range of output rows; each warp takes one row of the strip at a time, 8
// lanes per 128-channel block and 16 weights per lane: lane l of a block
// holds channels [8l, 8l+8) and [64+8l, 64+8l+8), so each 16-byte load or
// store of the warp covers four whole 128-byte segments. A group of 128 is
// one block; groups of 64 or 32 are one run of 8 or 4 lanes (the quantiser
// reduces each run separately). The strip's s and 1/s for a chunk of
// alphas are staged in shared memory once per block, in lane order (float4 q
// of lane l at [q][l]) so that every 16-byte shared load of a warp reads 512
// contiguous bytes without bank conflicts, and reused by every row. W is read
// once (the next row's weights are loaded while the current row runs through
// its alphas). Products, differences and the dequantisation run as packed
// fp32 pairs (one instruction, two correctly rounded results).

// Occupancy of the fake-quant kernel (build-time tunables, defaults measured best).
#ifndef AWQ_FQ_ALPHA_CHUNK
#define AWQ_FQ_ALPHA_CHUNK 20
#endif
#ifndef AWQ_FQ_BLOCKS_PER_SM
#define AWQ_FQ_BLOCKS_PER_SM 2
#endif
constexpr int kFqCols = 512;                       // input channels per strip (four 128-channel blocks)
constexpr int kFqWarps = 8;                        // rows in flight per block
constexpr int kFqAlphaChunk = AWQ_FQ_ALPHA_CHUNK;  // alphas staged in shared memory at once
constexpr int kFqSmem = 2 * kFqAlphaChunk * kFqCols * 4;  // s and 1/s: 80 KiB for 20 alphas
constexpr int kFqBlocksPerSm = AWQ_FQ_BLOCKS_PER_SM;

template <typename WT>
struct RowRegs;
template <>
struct RowRegs<uint16_t> {
  uint4 a, b;
  __device__ __forceinline__ void load(const uint16_t* p) {
    a = *reinterpret_cast<const uint4*>(p);
    b = *reinterpret_cast<const uint4*>(p + 64);
  }
  __device__ __forceinline__ void unpack(float2 (&w)[8]) const {
    const uint32_t x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = make_float2(bf16_lo(x[i]), bf16_hi(x[i]));
  }
};
template <>
struct RowRegs<float> {
  float4 a0, a1, b0, b1;
  __device__ __forceinline__ void load(const float* p) {
    a0 = *reinterpret_cast<const float4*>(p);
    a1 = *reinterpret_cast<const float4*>(p + 4);
    b0 = *reinterpret_cast<const float4*>(p + 64);
    b1 = *reinterpret_cast<const float4*>(p + 68);
  }
  __device__ __forceinline__ void unpack(float2 (&w)[8]) const {
    const float4 x[4] = {a0, a1, b0, b1};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[2 * i] = make_float2(x[i].x, x[i].y);
      w[2 * i + 1] = make_float2(x[i].z, x[i].w);
    }
  }
};

// The 16 values of one lane from a lane-ordered shared-memory row [4][32] of float4.
__device__ __forceinline__ void lds_lane16(const float4* row, int lane, float2 (&v)[8]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 x = row[q * 32 + lane];
    v[2 * q] = make_float2(x.x, x.y);
    v[2 * q + 1] = make_float2(x.z, x.w);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float2 v) { return pack_bf16x2(v.x, v.y); }

// Scales of one alpha for fq_lane16, from the lane-ordered shared-memory rows.
struct SmemLane {
  const float4* s;
  const float4* inv;
  int lane;
  __device__ __forceinline__ void load_s(float2 (&v)[8]) const { lds_lane16(s, lane, v); }
  __device__ __forceinline__ void load_inv(float2 (&v)[8]) const { lds_lane16(inv, lane, v); }
};

template <typename WT, bool REF, int GROUP>
__global__ void __launch_bounds__(kFqWarps * 32, kFqBlocksPerSm)
    fakequant_kernel(const WT* __restrict__ W, int N, int K, int G, const float* __restrict__ s,
                     const float* __restrict__ inv_s, float qmax, float floor_, int symmetric,
                     uint16_t* __restrict__ op, int64_t slot_elems, int nstrips, int rows_per_block) {
  extern __shared__ float4 fq_smem[];
  float4* ss = fq_smem;                          // [chunk][4][32] float4
  float4* si = fq_smem + kFqAlphaChunk * 128;    // same for 1/s
  const int strip = blockIdx.x % nstrips;
  const int col0 = strip * kFqCols;
  const int ncols = min(kFqCols, K - col0);  // a multiple of 128
  const int r_begin = (blockIdx.x / nstrips) * rows_per_block;
  const int r_end = min(N, r_begin + rows_per_block);
  if (r_begin >= r_end) return;  // uniform over the block
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 3, sub = lane & 7;
  // Groups past a partial strip repeat group 0's work and store nothing.
  const bool active = grp * 128 < ncols;
  const int slane = active ? lane : sub;
  const int c_lo = (active ? grp * 128 : 0) + sub * 8;  // channels c_lo + [0,8) and c_lo + 64 + [0,8)

  for (int a0 = 0; a0 < G; a0 += kFqAlphaChunk) {
    const int gc = min(kFqAlphaChunk, G - a0);
    __syncthreads();  // the previous chunk's scales are no longer read
    const int c4n = ncols >> 2;
    for (int i = threadIdx.x; i < gc * c4n; i += blockDim.x) {
      const int a = i / c4n, c4 = i - a * c4n;
      const int c = 4 * c4;  // channel within the strip -> (lane, float4 index q)
      const int e = c & 127, h = e & 63;
      const int ln = (c >> 7) * 8 + (h >> 3);
      const int q = (e >> 6) * 2 + ((h & 7) >> 2);
      const size_t g = (size_t)(a0 + a) * K + col0 + c;
      const bool ok = AWQ_IN(g, 4, (size_t)G * K);
      ss[(a * 4 + q) * 32 + ln] = ok ? *reinterpret_cast<const float4*>(s + g) : make_float4(1.f, 1.f, 1.f, 1.f);
      si[(a * 4 + q) * 32 + ln] = ok ? *reinterpret_cast<const float4*>(inv_s + g) : make_float4(1.f, 1.f, 1.f, 1.f);
    }
    __syncthreads();

    int row = r_begin + warp;
    RowRegs<WT> nxt{};
    [[maybe_unused]] const size_t wn = (size_t)N * K;  // elements of W and of one operand slot (bounds checks)
    if (row < r_end && AWQ_IN((size_t)row * K + col0 + c_lo, 72, wn)) nxt.load(W + (size_t)row * K + col0 + c_lo);
    for (; row < r_end; row += kFqWarps) {
      float2 w[8];
      nxt.unpack(w);
      const size_t base = (size_t)row * K + col0 + c_lo;
      if (row + kFqWarps < r_end && AWQ_IN(base + (size_t)kFqWarps * K, 72, wn))
        nxt.load(W + base + (size_t)kFqWarps * K);
      if (REF && a0 == 0 && active && AWQ_IN((size_t)G * slot_elems + base, 72, (size_t)(G + 1) * wn)) {
        uint4* dst = reinterpret_cast<uint4*>(op + (size_t)G * slot_elems + base);
        dst[0] = make_uint4(pack_bf16x2(w[0]), pack_bf16x2(w[1]), pack_bf16x2(w[2]), pack_bf16x2(w[3]));
        dst[8] = make_uint4(pack_bf16x2(w[4]), pack_bf16x2(w[5]), pack_bf16x2(w[6]), pack_bf16x2(w[7]));
      }
      float2 nw[8];  // -w
#pragma unroll
      for (int i = 0; i < 8; ++i) nw[i] = make_float2(-w[i].x, -w[i].y);
#pragma unroll 1
      for (int a = 0; a < gc; ++a) {
        uint32_t o[8];
        fq_lane16<REF, GROUP>(w, nw, SmemLane{ss + a * 128, si + a * 128, slane}, qmax, floor_, symmetric != 0, o);
        if (active && AWQ_IN((size_t)(a0 + a) * slot_elems + base, 72, (size_t)(REF ? G + 1 : G) * wn)) {
          uint4* dst = reinterpret_cast<uint4*>(op + (size_t)(a0 + a) * slot_elems + base);
          dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
          dst[8] = make_uint4(o[4], o[5], o[6], o[7]);  // 64 channels further on
        }
      }
    }
  }
}

template <typename WT, bool REF, int GROUP>
cudaError_t launch_fakequant_t(const WT* W, int64_t N, int64_t K, const float* s, const float* inv_s,
                               const awq_config& cfg, uint16_t* op, cudaStream_t st) {
  cudaError_t e = ensure_dynamic_smem((const void*)fakequant_kernel<WT, REF, GROUP>, kFqSmem);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  const int nstrips = (int)((K + kFqCols - 1) / kFqCols);
  // one wave: at most kFqBlocksPerSm blocks per SM in total
  int64_t rblocks = (int64_t)sms * kFqBlocksPerSm / nstrips;
  if (rblocks < 1) rblocks = 1;
  if (rblocks > N) rblocks = N;
  const int rows_per_block = (int)((N + rblocks - 1) / rblocks);
  rblocks = (N + rows_per_block - 1) / rows_per_block;
  const float qmax = (float)((1 << cfg.w_bit) - 1);
  fakequant_kernel<WT, REF, GROUP><<<(unsigned)(rblocks * nstrips), kFqWarps * 32, kFqSmem, st>>>(
      W, (int)N, (int)K, cfg.n_grid, s, inv_s, qmax, cfg.delta_floor, cfg.zero_point == 0 ? 1 : 0, op, N * K,
      nstrips, rows_per_block);
  return cudaGetLastError();
}

template <int GROUP>
cudaError_t launch_fakequant_g(const void* W, int w_dtype, int64_t N, int64_t K, const float* s,
                               const float* inv_s, const awq_config& cfg, uint16_t* op, cudaStream_t st) {
  const bool ref = cfg.loss_form == AWQ_LOSS_REFERENCE;
  if (w_dtype == AWQ_BF16) {
    const uint16_t* w = (const uint16_t*)W;
    return ref ? launch_fakequant_t<uint16_t, true, GROUP>(w, N, K, s, inv_s, cfg, op, st)
               : launch_fakequant_t<uint16_t, false, GROUP>(w, N, K, s, inv_s, cfg, op, st);
  }
  const float* w = (const float*)W;
  return ref ? launch_fakequant_t<float, true, GROUP>(w, N, K, s, inv_s, cfg, op, st)
             : launch_fakequant_t<float, false, GROUP>(w, N, K, s, inv_s, cfg, op, st);
}

cudaError_t launch_fakequant(const void* W, int w_dtype, int64_t N, int64_t K, const float* s,
                             const float* inv_s, const awq_config& cfg, uint16_t* op, cudaStream_t st) {
  switch (cfg.group) {
    case 32: return launch_fakequant_g<32>(W, w_dtype, N, K, s, inv_s, cfg, op, st);
    case 64: return launch_fakequant_g<64>(W, w_dtype, N, K, s, inv_s, cfg, op, st);
    case 128: return launch_fakequant_g<128>(W, w_dtype, N, K, s, inv_s, cfg, op, st);
    default: return cudaErrorInvalidValue;
  }
}

// ============================================================== pack
//
// Final codes of W * diag(s) with the same quantiser, 8 codes per int32
// ("What is AWQ Quantization? ...", "INT4 Weight Packing & Export"), one fp16
// scale ("AWQ (Activation-Aware Weight Quantization) - AI Glossary", memory
// example) and one fp16 zero per group. Same layout as the fake-quant
// kernel: a block owns a 512-channel strip and a row range, a warp one row at
// a time, 8 lanes per 128-channel block with channels [8l, 8l+8) and
// [64+8l, 64+8l+8), so lane l's two code words are words l and 8+l of its
// block and every 4-byte store instruction of a warp fills four whole 32-byte
// sectors. The
// lane's 16 scales are loaded once per block; the next row's weights load
// while the current row is quantised.

constexpr int kPackWarps = 8;
// resident blocks per SM: fp32 weights, and two groups per lane, need more
// registers than the 80 of three blocks
template <typename WT, int GROUP>
constexpr int pack_blocks_per_sm() { return (sizeof(WT) == 2 && GROUP == 128) ? 3 : 2; }

template <typename WT, int GROUP, int BITS>
__global__ void __launch_bounds__(kPackWarps * 32, pack_blocks_per_sm<WT, GROUP>())
    pack_kernel(const WT* __restrict__ W, int N, int K, const float* __restrict__ s, float qmax, float floor_,
                int symmetric, int32_t* __restrict__ qweight, uint16_t* __restrict__ scales,
                uint16_t* __restrict__ zeros, int nstrips, int rows_per_block) {
  const int strip = blockIdx.x % nstrips;
  const int col0 = strip * kFqCols;
  const int ncols = min(kFqCols, K - col0);
  const int r_begin = (blockIdx.x / nstrips) * rows_per_block;
  const int r_end = min(N, r_begin + rows_per_block);
  if (r_begin >= r_end) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 3, sub = lane & 7;
  const bool active = grp * 128 < ncols;  // blocks past a partial strip repeat block 0 and store nothing
  const int c_lo = (active ? grp * 128 : 0) + sub * 8;
  // the lane stores the scale and zero of each group whose first channel it
  // holds: run A's group when its run starts one, and (for groups under 128)
  // run B's group, 64 channels further on
  const bool lead = (sub % (GROUP / 8 < 8 ? GROUP / 8 : 8)) == 0;
  float2 sv[8];
  {
    float t[16] = {};
    if (AWQ_IN(col0 + c_lo, 72, K)) {
      load8f(s + col0 + c_lo, t);
      load8f(s + col0 + c_lo + 64, t + 8);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) sv[i] = make_float2(t[2 * i], t[2 * i + 1]);
  }
  const int kw = K * BITS / 32, kg = K / GROUP;  // code words and groups per row
  [[maybe_unused]] const size_t wn = (size_t)N * K;  // elements of W (bounds checks)
  int row = r_begin + warp;
  RowRegs<WT> nxt{};
  if (row < r_end && AWQ_IN((size_t)row * K + col0 + c_lo, 72, wn)) nxt.load(W + (size_t)row * K + col0 + c_lo);
  for (; row < r_end; row += kPackWarps) {
    float2 w[8];
    nxt.unpack(w);
    if (row + kPackWarps < r_end && AWQ_IN((size_t)(row + kPackWarps) * K + col0 + c_lo, 72, wn))
      nxt.load(W + (size_t)(row + kPackWarps) * K + col0 + c_lo);
    float2 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __fmul2_rn(w[i], sv[i]);
    GroupFast ga, gb;
    lane_groups<GROUP>(v, qmax, floor_, symmetric != 0, ga, gb);
    float2 k[8];
    lane_codes_minus_z<GROUP>(v, ga, gb, k);
    uint32_t wa[2] = {0u, 0u}, wb[2] = {0u, 0u};  // run A's and run B's words
    if constexpr (BITS == 4) {
      // q = (q - z) + z, exact integers in [0, 15]. A run of 8 codes is one word q_0 + 16 q_1 + ... + 16^7 q_7
      // (column order), built as two 16-bit halves h = (q_0 + 256 q_2) + 16 (q_1 + 256 q_3): every step is
      // exact in fp32 (h < 2^16), and 2^23 + h carries h in its low mantissa bits, so one byte permute joins
      // the two halves without a float-to-integer conversion or a shift per code
      const float2 za = make_float2(ga.z, ga.z), zb = make_float2(gb.z, gb.z);
      const float2 c256 = make_float2(256.0f, 256.0f);
      float2 qa4[4], qb4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        qa4[i] = __fadd2_rn(k[i], za);
        qb4[i] = __fadd2_rn(k[4 + i], zb);
      }
      const float2 pa0 = __ffma2_rn(qa4[1], c256, qa4[0]), pa1 = __ffma2_rn(qa4[3], c256, qa4[2]);
      const float2 pb0 = __ffma2_rn(qb4[1], c256, qb4[0]), pb1 = __ffma2_rn(qb4[3], c256, qb4[2]);
      const float ha0 = __fmaf_rn(pa0.y, 16.0f, __fadd_rn(pa0.x, 8388608.0f));
      const float ha1 = __fmaf_rn(pa1.y, 16.0f, __fadd_rn(pa1.x, 8388608.0f));
      const float hb0 = __fmaf_rn(pb0.y, 16.0f, __fadd_rn(pb0.x, 8388608.0f));
      const float hb1 = __fmaf_rn(pb1.y, 16.0f, __fadd_rn(pb1.x, 8388608.0f));
      wa[0] = __byte_perm(__float_as_uint(ha0), __float_as_uint(ha1), 0x5410);
      wb[0] = __byte_perm(__float_as_uint(hb0), __float_as_uint(hb1), 0x5410);
    } else {
      // q = (q - z) + z in [0, 2^b - 1]; 2^23 + q carries q in its low mantissa
      // bits, which avoids a float-to-integer conversion per code
      const float2 za = make_float2(8388608.0f + ga.z, 8388608.0f + ga.z);
      const float2 zb = make_float2(8388608.0f + gb.z, 8388608.0f + gb.z);
      constexpr uint32_t kMask = (1u << BITS) - 1u;
      uint32_t qa[8], qb[8];  // the codes of run A and run B
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = __fadd2_rn(k[i], za);
        const float2 b = __fadd2_rn(k[4 + i], zb);
        qa[2 * i] = __float_as_uint(a.x) & kMask;
        qa[2 * i + 1] = __float_as_uint(a.y) & kMask;
        qb[2 * i] = __float_as_uint(b.x) & kMask;
        qb[2 * i + 1] = __float_as_uint(b.y) & kMask;
      }
      // words of 32 / BITS codes, column (32/b) j + k in bits [b k, b k + b) of word j: a run of 8 codes is
      // two words (8 bits) or half a word (2 bits, joined with the next lane's half)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int word = (e * BITS) >> 5, bit = (e * BITS) & 31;
        wa[word] |= qa[e] << bit;
        wb[word] |= qb[e] << bit;
      }
      if (BITS == 2) {  // the odd lane's 16 bits go above the even lane's (8 channels further on)
        wa[0] |= __shfl_down_sync(0xffffffffu, wa[0], 1) << 16;
        wb[0] |= __shfl_down_sync(0xffffffffu, wb[0], 1) << 16;
      }
    }
    const size_t w_at = (size_t)row * kw + (size_t)(col0 + c_lo) * BITS / 32;  // run A's first word
    constexpr int kRunB = 64 * BITS / 32;                                      // words from run A to run B
    if (active && AWQ_IN(w_at, kRunB + (BITS == 8 ? 2 : 1), (size_t)N * kw)) {
      int32_t* q = qweight + w_at;
      if (BITS == 4) {
        q[0] = (int32_t)wa[0];
        q[kRunB] = (int32_t)wb[0];
      } else if (BITS == 8) {
        *reinterpret_cast<int2*>(q) = make_int2((int)wa[0], (int)wa[1]);
        *reinterpret_cast<int2*>(q + kRunB) = make_int2((int)wb[0], (int)wb[1]);
      } else if ((sub & 1) == 0) {
        q[0] = (int32_t)wa[0];
        q[kRunB] = (int32_t)wb[0];
      }
      const size_t gi = (size_t)row * kg + (col0 + c_lo) / GROUP;
      if (lead && AWQ_IN(gi, GROUP < 128 ? 64 / GROUP + 1 : 1, (size_t)N * kg)) {
        scales[gi] = __half_as_ushort(__float2half_rn(ga.delta));
        zeros[gi] = __half_as_ushort(__float2half_rn(ga.z));
        if (GROUP < 128) {
          scales[gi + 64 / GROUP] = __half_as_ushort(__float2half_rn(gb.delta));
          zeros[gi + 64 / GROUP] = __half_as_ushort(__float2half_rn(gb.z));
        }
      }
    }
  }
}

template <typename WT, int GROUP, int BITS>
cudaError_t launch_pack_t(const WT* W, int64_t N, int64_t K, const float* s, const awq_config& cfg,
                          int32_t* qweight, uint16_t* scales, uint16_t* zeros, cudaStream_t st) {
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  const int nstrips = (int)((K + kFqCols - 1) / kFqCols);
  int64_t rblocks = (int64_t)sms * pack_blocks_per_sm<WT, GROUP>() / nstrips;
  if (rblocks < 1) rblocks = 1;
  if (rblocks > N) rblocks = N;
  const int rows_per_block = (int)((N + rblocks - 1) / rblocks);
  rblocks = (N + rows_per_block - 1) / rows_per_block;
  const float qmax = (float)((1 << cfg.w_bit) - 1);
  pack_kernel<WT, GROUP, BITS><<<(unsigned)(rblocks * nstrips), kPackWarps * 32, 0, st>>>(
      W, (int)N, (int)K, s, qmax, cfg.delta_floor, cfg.zero_point == 0 ? 1 : 0, qweight, scales, zeros, nstrips,
      rows_per_block);
  return cudaGetLastError();
}

template <int GROUP, int BITS>
cudaError_t launch_pack_b(const void* W, int w_dtype, int64_t N, int64_t K, const float* s, const awq_config& cfg,
                          int32_t* qweight, uint16_t* scales, uint16_t* zeros, cudaStream_t st) {
  if (w_dtype == AWQ_BF16)
    return launch_pack_t<uint16_t, GROUP, BITS>((const uint16_t*)W, N, K, s, cfg, qweight, scales, zeros, st);
  return launch_pack_t<float, GROUP, BITS>((const float*)W, N, K, s, cfg, qweight, scales, zeros, st);
}

template <int GROUP>
cudaError_t launch_pack_g(const void* W, int w_dtype, int64_t N, int64_t K, const float* s, const awq_config& cfg,
                          int32_t* qweight, uint16_t* scales, uint16_t* zeros, cudaStream_t st) {
  switch (cfg.w_bit) {
    case 2: return launch_pack_b<GROUP, 2>(W, w_dtype, N, K, s, cfg, qweight, scales, zeros, st);
    case 4: return launch_pack_b<GROUP, 4>(W, w_dtype, N, K, s, cfg, qweight, scales, zeros, st);
    case 8: return launch_pack_b<GROUP, 8>(W, w_dtype, N, K, s, cfg, qweight, scales, zeros, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_pack(const void* W, int w_dtype, int64_t N, int64_t K, const float* s, const awq_config& cfg,
                        int32_t* qweight, uint16_t* scales, uint16_t* zeros, cudaStream_t st) {
  switch (cfg.group) {
    case 32: return launch_pack_g<32>(W, w_dtype, N, K, s, cfg, qweight, scales, zeros, st);
    case 64: return launch_pack_g<64>(W, w_dtype, N, K, s, cfg, qweight, scales, zeros, st);
    case 128: return launch_pack_g<128>(W, w_dtype, N, K, s, cfg, qweight, scales, zeros, st);
    default: return cudaErrorInvalidValue;
  }
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
  for (int64_t t = threadIdx.x; t < per_alpha; t += blockDim.x)
    if (AWQ_IN((size_t)a * per_alpha + t, 1, (size_t)gridDim.x * per_alpha)) acc += p[t];
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
  if (j < K && AWQ_IN((size_t)best_sh * K + j, 1, (size_t)G * K)) s_best[j] = s[(size_t)best_sh * K + j];
}

__global__ void __launch_bounds__(256) row_losses_kernel(const double* __restrict__ row_acc, size_t total,
                                                         double denom, float* __restrict__ row_losses) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x)
    row_losses[i] = (float)(row_acc[i] / denom);
}

cudaError_t launch_row_losses(const double* row_acc, int G, int64_t N, int64_t n_tok, float* row_losses,
                              cudaStream_t st) {
  const size_t total = (size_t)G * (size_t)N;
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  size_t blocks = (total + 255) / 256;
  if (blocks > (size_t)sms * 8) blocks = (size_t)sms * 8;
  row_losses_kernel<<<(unsigned)blocks, 256, 0, st>>>(row_acc, total, (double)n_tok * (double)N, row_losses);
  return cudaGetLastError();
}

cudaError_t launch_loss_select(const float* partials, int G, int64_t per_alpha, int64_t n_tok, int64_t N,
                               const float* s, int64_t K, float* losses, int32_t* best_idx, float* s_best,
                               uint32_t* status, cudaStream_t st) {
  loss_reduce_kernel<<<G, 256, 0, st>>>(partials, per_alpha, (double)n_tok * (double)N, losses, status);
  select_kernel<<<(unsigned)((K + 255) / 256), 256, 0, st>>>(losses, G, s, (int)K, best_idx, s_best);
  return cudaGetLastError();
}

#ifdef AWQ_CHECKED
cudaError_t take_oob_kernels(unsigned long long* out) { return take_oob_record(out); }

// One check that fails by construction, the offset one past an n-element
// buffer: it is counted and the write is skipped (the buffer stays intact).
__global__ void bounds_selftest_kernel(float* buf, int n) {
  if (threadIdx.x == 0 && AWQ_IN(n, 1, n)) buf[n] = 1.0f;
}

cudaError_t launch_bounds_selftest(float* buf, int n, cudaStream_t st) {
  bounds_selftest_kernel<<<1, 32, 0, st>>>(buf, n);
  return cudaGetLastError();
}
#endif

}  // namespace awq
