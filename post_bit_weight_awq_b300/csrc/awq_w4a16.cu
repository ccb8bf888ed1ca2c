// Product of activations with a packed AWQ layer (w4a16): y = x * W_hat^T,
// W_hat[r][k] = (q[r][k] - z[r][g]) * scale[r][g], for a few tokens at a
// time (the decode case of "AWQ: How Activation-Aware Quantization Saves
// 4-bit LLMs", "What do you actually deploy": decoding is memory-bound and
// reads the 4-bit codes, a quarter of the bytes of fp16 weights).
//
// The packed layer is streamed from HBM once; x (at most 8 tokens) is
// converted to fp32 and staged in shared memory. One CTA of 16 or 32 warps
// per SM; each warp owns one output row at a time and each lane 32
// consecutive codes (one 16-byte load, inside one group of 128) per step,
// four steps' loads issued before any is used. Codes become floats without conversion
// instructions: a byte permute places a nibble under the exponent bits of
// 2^23 (0x4B00_00qq = 2^23 + q exactly), and one packed subtraction of
// 2^23 + z gives (q - z, q' - z) for two neighbouring columns, exactly. The
// lane accumulates x * (q - z) as fp32 pairs, scales the 32-column sum by
// the group's fp16 step once, and the warp adds its lanes at the end of the
// row.
#include <cuda_fp16.h>

#include "awq_device.cuh"
#include "awq_launch.h"

namespace awq {
namespace {

// threads per CTA: more warps (more loads in flight) while the registers of
// the M token accumulators still fit without spilling
template <int M>
__host__ __device__ constexpr int w4_threads() { return M <= 2 ? 1024 : 512; }
constexpr int kW4Unroll = 4;  // 16-byte code loads in flight per lane

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 2^23 + nibble of byte b of v (v holds one nibble per byte).
__device__ __forceinline__ float nib_f(uint32_t v, int b) {
  return __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7440u + (uint32_t)b));
}

template <int M>
__global__ void __launch_bounds__(w4_threads<M>(), 1)
    w4a16_gemv_kernel(const uint16_t* __restrict__ x, int K, const int32_t* __restrict__ qweight,
                      const uint16_t* __restrict__ scales, const uint16_t* __restrict__ zeros, int N,
                      float* __restrict__ y) {
  extern __shared__ float4 w4_smem[];
  float* xs = reinterpret_cast<float*>(w4_smem);  // [M][K] fp32
  constexpr int kThreads = w4_threads<M>(), kWarps = kThreads / 32;
  for (int i = threadIdx.x; i < M * K / 8; i += kThreads) {
    const uint4 v = *reinterpret_cast<const uint4*>(x + (size_t)i * 8);
    float4 a, b;
    a.x = bf16_lo(v.x);
    a.y = bf16_hi(v.x);
    a.z = bf16_lo(v.y);
    a.w = bf16_hi(v.y);
    b.x = bf16_lo(v.z);
    b.y = bf16_hi(v.z);
    b.z = bf16_lo(v.w);
    b.w = bf16_hi(v.w);
    w4_smem[2 * i] = a;
    w4_smem[2 * i + 1] = b;
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunks = K >> 5;  // 32-code chunks per row
  const int kw = K >> 3, kg = K >> 7;
  for (int r = blockIdx.x * kWarps + warp; r < N; r += gridDim.x * kWarps) {
    const int32_t* qrow = qweight + (size_t)r * kw;
    float acc[M];
#pragma unroll
    for (int m = 0; m < M; ++m) acc[m] = 0.0f;
    for (int c0 = lane; c0 < chunks; c0 += 32 * kW4Unroll) {
      uint4 q[kW4Unroll];
#pragma unroll
      for (int u = 0; u < kW4Unroll; ++u)
        if (c0 + 32 * u < chunks) q[u] = ld_stream_v4(qrow + 4 * (c0 + 32 * u));
#pragma unroll
      for (int u = 0; u < kW4Unroll; ++u) {
        const int c = c0 + 32 * u;
        if (c >= chunks) break;
        const int k0 = c << 5;
        const int g = k0 >> 7;
        const float sc = __half2float(__ushort_as_half(scales[(size_t)r * kg + g]));
        const float zoff = 8388608.0f + __half2float(__ushort_as_half(zeros[(size_t)r * kg + g]));
        const float2 nz = make_float2(-zoff, -zoff);
        float2 part[M];
#pragma unroll
        for (int m = 0; m < M; ++m) part[m] = make_float2(0.0f, 0.0f);
        const uint32_t wd[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t lo = wd[j] & 0x0F0F0F0Fu;         // nibbles 0, 2, 4, 6: even columns
          const uint32_t hi = (wd[j] >> 4) & 0x0F0F0F0Fu;  // nibbles 1, 3, 5, 7: odd columns
#pragma unroll
          for (int b = 0; b < 4; b += 2) {
            // columns k0 + 8j + 2b .. + 3
            const float2 w01 = __fadd2_rn(make_float2(nib_f(lo, b), nib_f(hi, b)), nz);
            const float2 w23 = __fadd2_rn(make_float2(nib_f(lo, b + 1), nib_f(hi, b + 1)), nz);
#pragma unroll
            for (int m = 0; m < M; ++m) {
              const float4 xv = *reinterpret_cast<const float4*>(xs + (size_t)m * K + k0 + 8 * j + 2 * b);
              part[m] = __ffma2_rn(w01, make_float2(xv.x, xv.y), part[m]);
              part[m] = __ffma2_rn(w23, make_float2(xv.z, xv.w), part[m]);
            }
          }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = fmaf(sc, part[m].x + part[m].y, acc[m]);
      }
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float v = acc[m];
#pragma unroll
      for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == m) y[(size_t)m * N + r] = v;
    }
  }
}

template <int M>
cudaError_t launch_w4_t(const uint16_t* x, int64_t K, const int32_t* qweight, const uint16_t* scales,
                        const uint16_t* zeros, int64_t N, float* y, cudaStream_t st) {
  const int smem = (int)(M * K * 4);
  cudaError_t e = cudaFuncSetAttribute(w4a16_gemv_kernel<M>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  constexpr int kThreads = w4_threads<M>();
  int64_t grid = (N + kThreads / 32 - 1) / (kThreads / 32);
  if (grid > sms) grid = sms;
  w4a16_gemv_kernel<M><<<(unsigned)grid, kThreads, smem, st>>>(x, (int)K, qweight, scales, zeros, (int)N, y);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_w4a16_gemv(const uint16_t* x, int64_t M, int64_t K, const int32_t* qweight, const uint16_t* scales,
                              const uint16_t* zeros, int64_t N, float* y, cudaStream_t st) {
  switch (M) {
    case 1: return launch_w4_t<1>(x, K, qweight, scales, zeros, N, y, st);
    case 2: return launch_w4_t<2>(x, K, qweight, scales, zeros, N, y, st);
    case 3: return launch_w4_t<3>(x, K, qweight, scales, zeros, N, y, st);
    case 4: return launch_w4_t<4>(x, K, qweight, scales, zeros, N, y, st);
    case 5: return launch_w4_t<5>(x, K, qweight, scales, zeros, N, y, st);
    case 6: return launch_w4_t<6>(x, K, qweight, scales, zeros, N, y, st);
    case 7: return launch_w4_t<7>(x, K, qweight, scales, zeros, N, y, st);
    case 8: return launch_w4_t<8>(x, K, qweight, scales, zeros, N, y, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace awq
