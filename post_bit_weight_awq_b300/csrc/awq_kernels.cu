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
// range of output rows; each warp takes two rows of the strip at a time, one
// per half-warp, in the quad layout of awq_quant.cuh: the 4 lanes of a quad
// share a 128-channel block, lane quarter p holding the runs of 8 channels at
// 32 j + 8 p (j = 0..3), 32 weights per lane. Every 16-byte load or store of
// a warp then covers 64 contiguous bytes of each of the 8 (row, block)
// pairs. The strip's s and 1/s for a chunk of alphas are staged in shared
// memory once per block, in the order the lanes read them (the 16 lanes of a
// half-warp read 256 contiguous bytes per 16-byte load, the two halves the
// same addresses), and reused by every row. W is read once: the next row
// pair's weights load while the current pair runs through its alphas.

// Occupancy of the fake-quant kernel (build-time tunables, defaults measured best).
#ifndef AWQ_FQ_ALPHA_CHUNK
#define AWQ_FQ_ALPHA_CHUNK 20
#endif
#ifndef AWQ_FQ_BLOCKS_PER_SM
#define AWQ_FQ_BLOCKS_PER_SM 2
#endif
constexpr int kFqCols = 512;                       // input channels per strip (four 128-channel blocks)
constexpr int kFqWarps = 8;                        // row pairs in flight per block
constexpr int kFqAlphaChunk = AWQ_FQ_ALPHA_CHUNK;  // alphas staged in shared memory at once
constexpr int kFqQuadF4 = 128;                     // float4 of s (or 1/s) per alpha per strip
constexpr int kFqSmem = 2 * kFqAlphaChunk * kFqQuadF4 * 16;  // s and 1/s: 80 KiB for 20 alphas
constexpr int kFqBlocksPerSm = AWQ_FQ_BLOCKS_PER_SM;

// A lane's 32 weights of one row in the quad layout (runs at c, c+32, c+64, c+96).
template <typename WT>
struct QuadRow;
template <>
struct QuadRow<uint16_t> {
  uint4 r[4];
  __device__ __forceinline__ void load(const uint16_t* p) {
#pragma unroll
    for (int j = 0; j < 4; ++j) r[j] = *reinterpret_cast<const uint4*>(p + 32 * j);
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int j = 0; j < 4; ++j) r[j] = make_uint4(0u, 0u, 0u, 0u);
  }
  __device__ __forceinline__ void unpack_run(int j, float2 (&w)[4]) const {
    const uint32_t x[4] = {r[j].x, r[j].y, r[j].z, r[j].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = make_float2(bf16_lo(x[i]), bf16_hi(x[i]));
  }
  __device__ __forceinline__ void unpack(float2 (&w)[16]) const {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 w4[4];
      unpack_run(j, w4);
#pragma unroll
      for (int i = 0; i < 4; ++i) w[4 * j + i] = w4[i];
    }
  }
};
template <>
struct QuadRow<float> {
  float4 r[8];
  __device__ __forceinline__ void load(const float* p) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      r[2 * j] = *reinterpret_cast<const float4*>(p + 32 * j);
      r[2 * j + 1] = *reinterpret_cast<const float4*>(p + 32 * j + 4);
    }
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int j = 0; j < 8; ++j) r[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __device__ __forceinline__ void unpack_run(int j, float2 (&w)[4]) const {
    w[0] = make_float2(r[2 * j].x, r[2 * j].y);
    w[1] = make_float2(r[2 * j].z, r[2 * j].w);
    w[2] = make_float2(r[2 * j + 1].x, r[2 * j + 1].y);
    w[3] = make_float2(r[2 * j + 1].z, r[2 * j + 1].w);
  }
  __device__ __forceinline__ void unpack(float2 (&w)[16]) const {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      w[2 * j] = make_float2(r[j].x, r[j].y);
      w[2 * j + 1] = make_float2(r[j].z, r[j].w);
    }
  }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float2 v) { return pack_bf16x2(v.x, v.y); }

// Scales of one alpha for fq_quad, from the staged shared-memory rows
// [4 runs][2 halves of a run][16 quad slots] of float4.
struct SmemQuad {
  const float4* s;
  const float4* inv;
  int slot;  // 4 * block + quarter
  __device__ __forceinline__ static void get(const float4* base, int slot, int j, float2 (&v)[4]) {
    const float4 a = base[(2 * j) * 16 + slot];
    const float4 b = base[(2 * j + 1) * 16 + slot];
    v[0] = make_float2(a.x, a.y);
    v[1] = make_float2(a.z, a.w);
    v[2] = make_float2(b.x, b.y);
    v[3] = make_float2(b.z, b.w);
  }
  __device__ __forceinline__ void load_s(int j, float2 (&v)[4]) const { get(s, slot, j, v); }
  __device__ __forceinline__ void load_inv(int j, float2 (&v)[4]) const { get(inv, slot, j, v); }
};

template <typename WT, bool REF, int GROUP>
__global__ void __launch_bounds__(kFqWarps * 32, kFqBlocksPerSm)
    fakequant_kernel(const WT* __restrict__ W, int N, int K, int G, const float* __restrict__ s,
                     const float* __restrict__ inv_s, float qmax, float floor_, int symmetric,
                     uint16_t* __restrict__ op, int64_t slot_elems, int nstrips, int rows_per_block) {
  extern __shared__ float4 fq_smem[];
  float4* ss = fq_smem;                            // [chunk][4][2][16] float4
  float4* si = fq_smem + kFqAlphaChunk * kFqQuadF4;  // same for 1/s
  const int strip = blockIdx.x % nstrips;
  const int col0 = strip * kFqCols;
  const int ncols = min(kFqCols, K - col0);  // a multiple of 128
  const int r_begin = (blockIdx.x / nstrips) * rows_per_block;
  const int r_end = min(N, r_begin + rows_per_block);
  if (r_begin >= r_end) return;  // uniform over the block
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hw = lane >> 4, blk = (lane >> 2) & 3, quarter = lane & 3;
  // Blocks past a partial strip repeat block 0's work and store nothing.
  const bool active = blk * 128 < ncols;
  const int slot = (active ? blk : 0) * 4 + quarter;
  const int c_lo = (active ? blk * 128 : 0) + 8 * quarter;  // runs at c_lo + 32 j within the strip
  const QuantSpec q = make_quant_spec(qmax, floor_, symmetric != 0);
  [[maybe_unused]] const size_t wn = (size_t)N * K;  // elements of W and of one operand slot (bounds checks)
  const int pair_step = 2 * kFqWarps;

  for (int a0 = 0; a0 < G; a0 += kFqAlphaChunk) {
    const int gc = min(kFqAlphaChunk, G - a0);
    __syncthreads();  // the previous chunk's scales are no longer read
    for (int i = threadIdx.x; i < gc * kFqQuadF4; i += blockDim.x) {
      const int a = i / kFqQuadF4, c = 4 * (i - a * kFqQuadF4);  // channel within the strip
      const int b = c >> 7, e = c & 127;
      const int idx = ((a * 4 + (e >> 5)) * 2 + ((e & 7) >> 2)) * 16 + b * 4 + ((e & 31) >> 3);
      const size_t g = (size_t)(a0 + a) * K + col0 + c;
      const bool ok = c < ncols && AWQ_IN(g, 4, (size_t)G * K);
      ss[idx] = ok ? *reinterpret_cast<const float4*>(s + g) : make_float4(1.f, 1.f, 1.f, 1.f);
      si[idx] = ok ? *reinterpret_cast<const float4*>(inv_s + g) : make_float4(1.f, 1.f, 1.f, 1.f);
    }
    __syncthreads();

    // row pairs: this half-warp's row is first + hw; the loop condition is the pair's, uniform over the warp.
    // A pair's weights are loaded as it starts: its alpha loop is long, and the other warps of the SM issue
    // while this one waits, so a prefetch buffer would only cost registers.
    for (int first = r_begin + 2 * warp; first < r_end; first += pair_step) {
      const int row = first + hw;
      const bool live = row < r_end;
      const size_t base = (size_t)row * K + col0 + c_lo;
      float2 w[16];
      {
        QuadRow<WT> cur;
        cur.zero();
        if (live && AWQ_IN(base, 104, wn)) cur.load(W + base);
        cur.unpack(w);
      }
      if (REF && a0 == 0 && live && active && AWQ_IN((size_t)G * slot_elems + base, 104, (size_t)(G + 1) * wn)) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(op + (size_t)G * slot_elems + base + 32 * j) =
              make_uint4(pack_bf16x2(w[4 * j]), pack_bf16x2(w[4 * j + 1]), pack_bf16x2(w[4 * j + 2]),
                         pack_bf16x2(w[4 * j + 3]));
      }
#pragma unroll 1
      for (int a = 0; a < gc; ++a) {
        const bool store =
            live && active && AWQ_IN((size_t)(a0 + a) * slot_elems + base, 104, (size_t)(REF ? G + 1 : G) * wn);
        fq_quad<REF, GROUP>(w, SmemQuad{ss + a * kFqQuadF4, si + a * kFqQuadF4, slot}, q,
                            op + (size_t)(a0 + a) * slot_elems + base, store);
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
// kernel: a block owns a 512-channel strip and a row range, a warp two rows
// at a time (one per half-warp) in the quad layout, so a lane's run j of 8
// channels is one 4-bit code word (words 16 block + 4 j + quarter of the
// strip's row) and the 4 lanes of a quad write 16 contiguous bytes per
// store instruction. The strip's scales are staged in shared memory once
// per block. The weights go through a per-warp ring of kPackStages row pairs
// in shared memory, filled by per-thread asynchronous copies: each lane
// copies the 4 runs it will read, so no lane waits on another, and two row
// pairs are in flight while the third is quantised (the arithmetic takes
// about a third of the issue slots, so the bytes in flight set the speed).

constexpr int kPackWarps = 8;
#ifndef AWQ_PACK_STAGES
#define AWQ_PACK_STAGES 3
#endif
constexpr int kPackStages = AWQ_PACK_STAGES;  // row pairs per warp in the shared-memory ring (build-time tunable)
template <typename WT>
constexpr int pack_pieces() { return 4 * (int)sizeof(WT) / 2; }  // 16-byte pieces of a lane's 32 weights
template <typename WT>
constexpr int pack_ring_bytes() { return kPackWarps * kPackStages * pack_pieces<WT>() * 32 * 16; }
// resident blocks per SM for bf16 weights in groups of 128 (build-time tunable); fp32 weights, and several
// groups per lane, need more registers and run 2
#ifndef AWQ_PACK_BLOCKS_PER_SM
#define AWQ_PACK_BLOCKS_PER_SM 3
#endif
template <typename WT, int GROUP>
constexpr int pack_blocks_per_sm() { return (sizeof(WT) == 2 && GROUP == 128) ? AWQ_PACK_BLOCKS_PER_SM : 2; }

// Code word(s) of one run of 8 codes k + z (k = q - z as fp32 pairs, exact small integers).
// BITS 4: one word, q_0 + 16 q_1 + ... + 16^7 q_7, built as two 16-bit halves
// (q_0 + 256 q_2) + 16 (q_1 + 256 q_3): every step is exact in fp32 (each half
// < 2^16), and 2^23 + half carries the half in its low mantissa bits, so one
// byte permute joins the halves without a float-to-integer conversion or a
// shift per code. BITS 8: two words of 4 codes; BITS 2: the low 16 bits of a
// word (the run's 8 codes), joined with the next run's by the caller.
template <int BITS>
__device__ __forceinline__ void run_words(const float2 (&k)[4], float z, uint32_t (&wd)[2]) {
  const float2 zz = make_float2(z, z);
  float2 qf[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) qf[i] = __fadd2_rn(k[i], zz);
  if constexpr (BITS == 4) {
    const float2 c256 = make_float2(256.0f, 256.0f);
    const float2 p0 = __ffma2_rn(qf[1], c256, qf[0]), p1 = __ffma2_rn(qf[3], c256, qf[2]);
    const float h0 = __fmaf_rn(p0.y, 16.0f, __fadd_rn(p0.x, 8388608.0f));
    const float h1 = __fmaf_rn(p1.y, 16.0f, __fadd_rn(p1.x, 8388608.0f));
    wd[0] = __byte_perm(__float_as_uint(h0), __float_as_uint(h1), 0x5410);
    wd[1] = 0u;
  } else {
    // 2^23 + q carries q in its low mantissa bits
    constexpr uint32_t kMask = (1u << BITS) - 1u;
    wd[0] = 0u;
    wd[1] = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = __fadd2_rn(qf[i], make_float2(8388608.0f, 8388608.0f));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = 2 * i + h;
        const uint32_t code = __float_as_uint(h ? a.y : a.x) & kMask;
        wd[(e * BITS) >> 5] |= code << ((e * BITS) & 31);
      }
    }
  }
}

// The 8 weights of one run as fp32 pairs (bf16 or fp32 storage).
__device__ __forceinline__ void load_run(const uint16_t* p, float2 (&w)[4]) {
  const uint4 r = *reinterpret_cast<const uint4*>(p);
  const uint32_t x[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = make_float2(bf16_lo(x[i]), bf16_hi(x[i]));
}
__device__ __forceinline__ void load_run(const float* p, float2 (&w)[4]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  w[0] = make_float2(a.x, a.y);
  w[1] = make_float2(a.z, a.w);
  w[2] = make_float2(b.x, b.y);
  w[3] = make_float2(b.z, b.w);
}

template <typename WT, int GROUP, int BITS>
__global__ void __launch_bounds__(kPackWarps * 32, pack_blocks_per_sm<WT, GROUP>())
    pack_kernel(const WT* __restrict__ W, int N, int K, const float* __restrict__ s, float qmax, float floor_,
                int symmetric, int32_t* __restrict__ qweight, uint16_t* __restrict__ scales,
                uint16_t* __restrict__ zeros, int nstrips, int rows_per_block) {
  constexpr int NG = quad_groups<GROUP>(), RUNS = 4 / NG;  // groups per lane, runs per group
  const int strip = blockIdx.x % nstrips;
  const int col0 = strip * kFqCols;
  const int ncols = min(kFqCols, K - col0);
  const int r_begin = (blockIdx.x / nstrips) * rows_per_block;
  const int r_end = min(N, r_begin + rows_per_block);
  if (r_begin >= r_end) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hw = lane >> 4, blk = (lane >> 2) & 3, quarter = lane & 3;
  const bool active = blk * 128 < ncols;  // blocks past a partial strip repeat block 0 and store nothing
  const int c_lo = (active ? blk * 128 : 0) + 8 * quarter;  // runs at c_lo + 32 j within the strip
  const QuantSpec q = make_quant_spec(qmax, floor_, symmetric != 0);
  // the strip's scales in shared memory, in the order the lanes read them (as the fake-quant kernel stages
  // one alpha); registers hold the weights in flight instead
  __shared__ float4 s_sm[kFqQuadF4];
  for (int i = threadIdx.x; i < kFqQuadF4; i += blockDim.x) {
    const int c = 4 * i, b = c >> 7, e = c & 127;
    const int idx = ((e >> 5) * 2 + ((e & 7) >> 2)) * 16 + b * 4 + ((e & 31) >> 3);
    s_sm[idx] = c < ncols && AWQ_IN(col0 + c, 4, K) ? *reinterpret_cast<const float4*>(s + col0 + c)
                                                    : make_float4(1.f, 1.f, 1.f, 1.f);
  }
  __syncthreads();
  const int slot = (active ? blk : 0) * 4 + quarter;
  const int kw = K * BITS / 32, kg = K / GROUP;  // code words and groups per row
  [[maybe_unused]] const size_t wn = (size_t)N * K;  // elements of W (bounds checks)
  const int pair_step = 2 * kPackWarps;
  // the warp's ring (dynamic shared memory): [stage][16-byte piece][lane] (a lane's 4 runs are 4 pieces of
  // bf16, 8 of fp32)
  constexpr int kPieces = pack_pieces<WT>();
  extern __shared__ uint4 pack_ring[];
  uint4* ring = pack_ring + (size_t)warp * kPackStages * kPieces * 32 + lane;
  // copy the lane's runs of row pair `it` into its stage (zeros past the last row)
  auto fetch = [&](int it) {
    const int row = r_begin + 2 * warp + it * pair_step + hw;
    uint4* dst = ring + (it % kPackStages) * kPieces * 32;
    if (row < r_end && AWQ_IN((size_t)row * K + col0 + c_lo, 104, wn)) {
      const uint8_t* src = reinterpret_cast<const uint8_t*>(W + (size_t)row * K + col0 + c_lo);
#pragma unroll
      for (int pc = 0; pc < kPieces; ++pc)
        cp_async16(dst + pc * 32, src + (pc / (kPieces / 4)) * 32 * sizeof(WT) + (pc % (kPieces / 4)) * 16);
    } else {
#pragma unroll
      for (int pc = 0; pc < kPieces; ++pc) dst[pc * 32] = make_uint4(0u, 0u, 0u, 0u);
    }
    cp_async_commit();
  };
  // run j's 4 pairs of weights from the stage of row pair `it`
  auto run_of = [&](int it, int j, float2 (&w4)[4]) {
    const uint4* src = ring + (it % kPackStages) * kPieces * 32;
    if constexpr (sizeof(WT) == 2) {
      const uint4 r = src[j * 32];
      const uint32_t x[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) w4[i] = make_float2(bf16_lo(x[i]), bf16_hi(x[i]));
    } else {
      const uint4 a = src[(2 * j) * 32], b = src[(2 * j + 1) * 32];
      w4[0] = make_float2(__uint_as_float(a.x), __uint_as_float(a.y));
      w4[1] = make_float2(__uint_as_float(a.z), __uint_as_float(a.w));
      w4[2] = make_float2(__uint_as_float(b.x), __uint_as_float(b.y));
      w4[3] = make_float2(__uint_as_float(b.z), __uint_as_float(b.w));
    }
  };
  const int npairs = (r_end - r_begin - 2 * warp + pair_step - 1) / pair_step;  // this warp's row pairs
#pragma unroll
  for (int it = 0; it < kPackStages - 1; ++it) fetch(it);
  for (int it = 0; it < npairs; ++it) {
    cp_async_wait<kPackStages - 2>();  // row pair `it` has landed (this lane's copies)
    fetch(it + kPackStages - 1);       // into the stage row pair it - 1 used
    const int row = r_begin + 2 * warp + it * pair_step + hw;
    const bool live = row < r_end && active;
    float2 v[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 w4[4], sv[4];
      run_of(it, j, w4);
      SmemQuad::get(s_sm, slot, j, sv);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[4 * j + i] = __fmul2_rn(w4[i], sv[i]);
    }
    GroupFast g[NG];
    quad_group_params<GROUP>(v, q, g);
    // codes in place; a group redone by division (rare) forms its values again from the stage
    quad_codes<GROUP>(v, g, [&](int j, float2 (&v4)[4]) {
      float2 w4[4], sv[4];
      run_of(it, j, w4);
      SmemQuad::get(s_sm, slot, j, sv);
#pragma unroll
      for (int i = 0; i < 4; ++i) v4[i] = __fmul2_rn(w4[i], sv[i]);
    });
    uint32_t words[4][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 k4[4] = {v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]};
      run_words<BITS>(k4, g[j / RUNS].z, words[j]);
    }
    if (BITS == 2) {  // the odd quarter's 16 bits go above the even quarter's (8 channels further on)
#pragma unroll
      for (int j = 0; j < 4; ++j) words[j][0] |= __shfl_down_sync(0xffffffffu, words[j][0], 1) << 16;
    }
    if (live) {
      const size_t w_row = (size_t)row * kw + (size_t)(col0 + c_lo) * BITS / 32;  // run 0's first word
      constexpr int kRunWords = 32 * BITS / 32;                                   // words from run j to j + 1
      if (AWQ_IN(w_row, 3 * kRunWords + (BITS == 8 ? 2 : 1), (size_t)N * kw)) {
        int32_t* dst = qweight + w_row;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (BITS == 8)
            *reinterpret_cast<int2*>(dst + j * kRunWords) = make_int2((int)words[j][0], (int)words[j][1]);
          else if (BITS == 4 || (quarter & 1) == 0)
            dst[j * kRunWords] = (int32_t)words[j][0];
        }
      }
      // the quarter holding each group's first channel stores its fp16 step and zero
      const size_t gi0 = (size_t)row * kg + (col0 + c_lo) / GROUP;
      if (quarter == 0 && AWQ_IN(gi0, NG, (size_t)N * kg)) {
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
          scales[gi0 + gi] = __half_as_ushort(__float2half_rn(g[gi].delta));
          zeros[gi0 + gi] = __half_as_ushort(__float2half_rn(g[gi].z));
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
  e = ensure_dynamic_smem((const void*)pack_kernel<WT, GROUP, BITS>, pack_ring_bytes<WT>());
  if (e != cudaSuccess) return e;
  pack_kernel<WT, GROUP, BITS><<<(unsigned)(rblocks * nstrips), kPackWarps * 32, pack_ring_bytes<WT>(), st>>>(
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
