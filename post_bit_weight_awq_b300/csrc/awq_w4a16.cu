// Product of activations with a packed AWQ layer (w4a16): y = x * W_hat^T,
// W_hat[r][k] = (q[r][k] - z[r][g]) * scale[r][g], for a few tokens at a
// time (the decode case of "AWQ: How Activation-Aware Quantization Saves
// 4-bit LLMs", "What do you actually deploy": decoding is memory-bound and
// reads the 4-bit codes, a quarter of the bytes of fp16 weights).
//
// The packed layer is streamed from HBM once; x (at most 8 tokens) is
// converted to fp32 and staged in shared memory. One CTA of 16 warps per SM;
// each warp owns R output rows at a time and each lane 4 / R chunks of 32
// consecutive codes of each (16-byte loads, each inside one group)
// per step, with the next step's loads in flight while the current one is
// computed. Codes become floats without conversion
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

constexpr int kW4Threads = 512;
constexpr int kW4Warps = kW4Threads / 32;
constexpr int kW4Pad = 36;    // shared-memory floats per 32 channels of x

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

// A step of a warp covers R rows and U chunks of 32 codes per lane (lane l
// takes chunks base + l + 32u of each of the R rows): R * U = 4 16-byte code
// loads per lane, and the next step's loads are in flight while the current
// one is computed. The lane's x values of a chunk (32 per token) are read
// from shared memory once and used for all R rows, which divides the
// shared-memory traffic (4 bytes of x per 4-bit code) by R. The launcher
// takes, among the R the registers allow (up to 4 for one token, 2 for two,
// else 1), the one that leaves the fewest warps idle in the last round of
// row groups; U = 4 / R (2 for more than four tokens).
template <int M>
__host__ __device__ constexpr int w4_max_rows() { return M == 1 ? 4 : (M == 2 ? 2 : 1); }

template <int R, int U>
struct W4Step {
  uint4 q[R][U];
  uint16_t s[R][U], z[R][U];
};

template <int R, int U>
__device__ __forceinline__ void w4_load(W4Step<R, U>& st, const int32_t* __restrict__ qweight,
                                        const uint16_t* __restrict__ scales, const uint16_t* __restrict__ zeros,
                                        int r0, int N, int cbase, int chunks, int kw, int kg, int gsh) {
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int r = r0 + i;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = cbase + 32 * u;
      if (r < N && c < chunks && AWQ_IN((size_t)r * kw + 4 * c, 4, (size_t)N * kw) &&
          AWQ_IN((size_t)r * kg + (c >> gsh), 1, (size_t)N * kg)) {
        st.q[i][u] = ld_stream_v4(qweight + (size_t)r * kw + 4 * c);
        st.s[i][u] = scales[(size_t)r * kg + (c >> gsh)];  // a chunk lies inside one group
        st.z[i][u] = zeros[(size_t)r * kg + (c >> gsh)];
      }
    }
  }
}

// x * (q - z) over the lane's 32 codes of one chunk: fp32 pairs, two columns at a time.
template <int M>
__device__ __forceinline__ void w4_chunk(const uint4 q, float zf, const float* __restrict__ xc, int kp, float2 (&part)[M]) {
  const float zoff = 8388608.0f + zf;
  const float2 nz = make_float2(-zoff, -zoff);
  const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = wd[j] & 0x0F0F0F0Fu;         // nibbles 0, 2, 4, 6: even columns
    const uint32_t hi = (wd[j] >> 4) & 0x0F0F0F0Fu;  // nibbles 1, 3, 5, 7: odd columns
#pragma unroll
    for (int b = 0; b < 4; b += 2) {
      // columns 8j + 2b .. + 3 of the chunk
      const float2 w01 = __fadd2_rn(make_float2(nib_f(lo, b), nib_f(hi, b)), nz);
      const float2 w23 = __fadd2_rn(make_float2(nib_f(lo, b + 1), nib_f(hi, b + 1)), nz);
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float4 xv = *reinterpret_cast<const float4*>(xc + (size_t)m * kp + 8 * j + 2 * b);
        part[m] = __ffma2_rn(w01, make_float2(xv.x, xv.y), part[m]);
        part[m] = __ffma2_rn(w23, make_float2(xv.z, xv.w), part[m]);
      }
    }
  }
}

template <int M, int R>
__global__ void __launch_bounds__(kW4Threads, 1)
    w4a16_gemv_kernel(const uint16_t* __restrict__ x, int K, const int32_t* __restrict__ qweight,
                      const uint16_t* __restrict__ scales, const uint16_t* __restrict__ zeros, int N, int gsh,
                      float* __restrict__ y) {
  constexpr int U = M > 4 ? 2 : 4 / R;  // fewer chunks in flight when many token accumulators need registers
  extern __shared__ float4 w4_smem[];
  // x as fp32, each run of 32 channels followed by 4 floats of padding: lane
  // l reads the run of chunk 32u + l, and the padding puts the 32 lanes'
  // 16-byte reads at the same offset into 8 distinct bank groups
  float* xs = reinterpret_cast<float*>(w4_smem);  // [M][K / 32][36]
  const int kp = (K >> 5) * kW4Pad;                // padded floats per token
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunks = K >> 5;  // 32-code chunks per row
  const int kw = K >> 3, kg = K >> (5 + gsh);  // groups of 32 << gsh codes
  const int steps_per_group = (chunks + 32 * U - 1) / (32 * U);
  const int gstride = gridDim.x * kW4Warps * R;

  // The warp's steps run through (group of R rows, step of U chunks); the
  // first step's loads go out before x is staged, so their latency overlaps it.
  int r0 = (blockIdx.x * kW4Warps + warp) * R, k = 0;
  W4Step<R, U> cur, nxt;
  if (r0 < N) w4_load<R, U>(cur, qweight, scales, zeros, r0, N, lane, chunks, kw, kg, gsh);

  for (int i = threadIdx.x; i < M * K / 8; i += kW4Threads) {
    const uint4 v = AWQ_IN((size_t)i * 8, 8, (size_t)M * K) ? *reinterpret_cast<const uint4*>(x + (size_t)i * 8)
                                                              : make_uint4(0u, 0u, 0u, 0u);
    const int m = (i * 8) / K, kk = i * 8 - m * K;
    float* d = xs + (size_t)m * kp + (kk >> 5) * kW4Pad + (kk & 31);
    reinterpret_cast<float4*>(d)[0] = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
    reinterpret_cast<float4*>(d)[1] = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
  }
  __syncthreads();

  float acc[R][M];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[i][m] = 0.0f;
  while (r0 < N) {
    int nr = r0, nk = k + 1;
    if (nk == steps_per_group) {
      nr = r0 + gstride;
      nk = 0;
    }
    if (nr < N) w4_load<R, U>(nxt, qweight, scales, zeros, nr, N, nk * 32 * U + lane, chunks, kw, kg, gsh);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = k * 32 * U + lane + 32 * u;
      if (c >= chunks) break;
      const float* xc = xs + c * kW4Pad;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        if (r0 + i >= N) break;
        float2 part[M];
#pragma unroll
        for (int m = 0; m < M; ++m) part[m] = make_float2(0.0f, 0.0f);
        w4_chunk<M>(cur.q[i][u], __half2float(__ushort_as_half(cur.z[i][u])), xc, kp, part);
        const float sc = __half2float(__ushort_as_half(cur.s[i][u]));
#pragma unroll
        for (int m = 0; m < M; ++m) acc[i][m] = fmaf(sc, part[m].x + part[m].y, acc[i][m]);
      }
    }
    if (nk == 0) {  // rows r0 .. r0 + R - 1 are complete
#pragma unroll
      for (int i = 0; i < R; ++i)
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float v = acc[i][m];
#pragma unroll
          for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == m && r0 + i < N && AWQ_IN((size_t)m * N + r0 + i, 1, (size_t)M * N)) y[(size_t)m * N + r0 + i] = v;
          acc[i][m] = 0.0f;
        }
    }
    cur = nxt;
    r0 = nr;
    k = nk;
  }
}

// ------------------------------------------------------------ prefill: expand, then the tensor-core product
//
// For token counts past the decode kernel's, the packed layer is expanded
// once to W_hat = bf16((q - z) * scale) (the fp32 product is exact: q - z is
// a small integer and the fp16 step has 11 significant bits) and multiplied
// with x on the tensor cores by the search kernels' CTA-pair product with
// G = 1 and its raw-product output. One thread expands one 32-bit word (8
// codes of one group) into 16 bytes.
__global__ void __launch_bounds__(256) w4_expand_kernel(const int32_t* __restrict__ qweight,
                                                        const uint16_t* __restrict__ scales,
                                                        const uint16_t* __restrict__ zeros, int64_t words, int kw,
                                                        int kg, int gsh, uint16_t* __restrict__ w_hat) {
  for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < words; w += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = w / kw;
    const int c = (int)(w - r * kw);               // word within the row: codes 8c .. 8c + 7
    const size_t gi = (size_t)r * kg + (c >> (gsh + 2));  // 8c / (32 << gsh)
    if (!AWQ_IN(w, 1, words) || !AWQ_IN(gi, 1, (size_t)(words / kw) * kg)) continue;
    const uint32_t q = (uint32_t)qweight[w];
    const float sc = __half2float(__ushort_as_half(scales[gi]));
    const float z = __half2float(__ushort_as_half(zeros[gi]));
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = __fmul_rn(__fsub_rn((float)((q >> (8 * j)) & 0xFu), z), sc);
      const float b = __fmul_rn(__fsub_rn((float)((q >> (8 * j + 4)) & 0xFu), z), sc);
      o[j] = pack_bf16x2(a, b);
    }
    if (AWQ_IN((size_t)w * 8, 8, (size_t)words * 8))
      *reinterpret_cast<uint4*>(w_hat + (size_t)w * 8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

template <int M, int R>
cudaError_t launch_w4_r(const uint16_t* x, int64_t K, const int32_t* qweight, const uint16_t* scales,
                        const uint16_t* zeros, int64_t N, int gsh, float* y, int sms, cudaStream_t st) {
  const int smem = (int)(M * (K / 32) * kW4Pad * 4);
  cudaError_t e = ensure_dynamic_smem((const void*)w4a16_gemv_kernel<M, R>, smem);
  if (e != cudaSuccess) return e;
  int64_t grid = (N + kW4Warps * R - 1) / (kW4Warps * R);
  if (grid > sms) grid = sms;
  w4a16_gemv_kernel<M, R><<<(unsigned)grid, kW4Threads, smem, st>>>(x, (int)K, qweight, scales, zeros, (int)N, gsh,
                                                                    y);
  return cudaGetLastError();
}

template <int M>
cudaError_t launch_w4_t(const uint16_t* x, int64_t K, const int32_t* qweight, const uint16_t* scales,
                        const uint16_t* zeros, int64_t N, int gsh, float* y, cudaStream_t st) {
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  // rows per warp: the candidate whose last round of row groups leaves the
  // fewest warps idle, unless a larger R (more reuse of x) is within 0.1 of it
  const int64_t warps = (int64_t)sms * kW4Warps;
  int R = 1;
  double best = -1.0;
  for (int r = w4_max_rows<M>(); r >= 1; r >>= 1) {
    const int64_t groups = (N + r - 1) / r;
    const int64_t rounds = (groups + warps - 1) / warps;
    const double busy = (double)groups / (double)(rounds * warps);
    if (busy > best + 0.1) {
      best = busy;
      R = r;
    }
  }
  if (R == 4)
    return launch_w4_r<M, (w4_max_rows<M>() >= 4 ? 4 : 1)>(x, K, qweight, scales, zeros, N, gsh, y, sms, st);
  if (R == 2)
    return launch_w4_r<M, (w4_max_rows<M>() >= 2 ? 2 : 1)>(x, K, qweight, scales, zeros, N, gsh, y, sms, st);
  return launch_w4_r<M, 1>(x, K, qweight, scales, zeros, N, gsh, y, sms, st);
}

}  // namespace

cudaError_t launch_w4_expand(const int32_t* qweight, const uint16_t* scales, const uint16_t* zeros, int64_t N,
                             int64_t K, int group, uint16_t* w_hat, cudaStream_t st) {
  const int gsh = group == 32 ? 0 : (group == 64 ? 1 : (group == 128 ? 2 : -1));
  if (gsh < 0) return cudaErrorInvalidValue;
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  const int64_t words = N * (K / 8);
  int64_t blocks = (words + 255) / 256;
  if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
  w4_expand_kernel<<<(unsigned)blocks, 256, 0, st>>>(qweight, scales, zeros, words, (int)(K / 8), (int)(K / group),
                                                      gsh, w_hat);
  return cudaGetLastError();
}

cudaError_t launch_w4a16_gemv(const uint16_t* x, int64_t M, int64_t K, const int32_t* qweight, const uint16_t* scales,
                              const uint16_t* zeros, int64_t N, int group, float* y, cudaStream_t st) {
  const int gsh = group == 32 ? 0 : (group == 64 ? 1 : (group == 128 ? 2 : -1));
  if (gsh < 0) return cudaErrorInvalidValue;
  switch (M) {
    case 1: return launch_w4_t<1>(x, K, qweight, scales, zeros, N, gsh, y, st);
    case 2: return launch_w4_t<2>(x, K, qweight, scales, zeros, N, gsh, y, st);
    case 3: return launch_w4_t<3>(x, K, qweight, scales, zeros, N, gsh, y, st);
    case 4: return launch_w4_t<4>(x, K, qweight, scales, zeros, N, gsh, y, st);
    case 5: return launch_w4_t<5>(x, K, qweight, scales, zeros, N, gsh, y, st);
    case 6: return launch_w4_t<6>(x, K, qweight, scales, zeros, N, gsh, y, st);
    case 7: return launch_w4_t<7>(x, K, qweight, scales, zeros, N, gsh, y, st);
    case 8: return launch_w4_t<8>(x, K, qweight, scales, zeros, N, gsh, y, st);
    default: return cudaErrorInvalidValue;
  }
}

#ifdef AWQ_CHECKED
cudaError_t take_oob_w4a16(unsigned long long* out) { return take_oob_record(out); }
#endif

}  // namespace awq
