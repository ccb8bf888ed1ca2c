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

#include "awq.h"
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

// ------------------------------------------------------------ decode on the tensor cores (groups of 128)
//
// The same product for groups of 128 with mma.sync (bf16 in, fp32
// accumulate; m16n8k16): a warp computes 16 output rows for all M <= 8
// tokens (the 8 columns of the MMA). Inside each group of 128 channels the
// order of k is permuted, the same way for the weights (A) and the
// activations (B), which leaves the dot product unchanged: thread quarter c
// of the MMA takes the group's channels 32 c .. 32 c + 31, i.e. 16 bytes of
// each of its two rows, and step kb = 2 m + h of the group pairs the codes
// (n_2h, n_2h+4) and (n_2h+1, n_2h+5) of word m. So
// (w >> 4j) & 0x000F000F | 0x43004300 is the bf16 pair (128 + n_j,
// 128 + n_j+4) in one mask-and-or, and one packed bf16 subtraction of
// 128 + z gives (q - z) exactly (small integers are exact in bf16). x is
// staged in shared memory once per block in the matching order: word j of
// each 8 consecutive channels holds channels j and j + 4, so one 16-byte load
// of x gives one 16-byte chunk of the staged words. Each (group, quarter) row
// of 16 words is padded to 20, so the four quarters' reads of one token fall
// in distinct banks. The MMA
// adds exact products in fp32; after the group's 8 MMAs the partial is
// scaled by the group's fp16 step and added to one of four running sums (in
// a fixed rotation, none taking more than a third of the groups), which are
// added at the end: every operation on the way keeps the error within a few
// dozen fp32 roundings of sum |x| |w| plus one per three groups.
// A zero point outside [-128, 127] (never produced for groups that contain
// both signs) is split as z = z_lo + 256 k, and the group takes one more MMA
// with the constant -256 k.
//
// A step of a warp covers two consecutive groups of its 16 rows: 16 MMAs in
// two independent chains. The codes stream through a per-warp ring of
// kMmaStages steps in shared memory, filled by per-thread asynchronous
// copies (each thread copies the 16-byte pieces of its two rows that it
// reads itself, so no thread waits on another). Rows past the layer's end
// are not copied: their sums land in output rows that are never stored.
// Each lane of a quad also loads one of its rows' steps or zeros for both
// groups of the step in one 4-byte load. The zero lanes pack both groups'
// bf16 128 + z_lo into one word and the step lanes pass their two fp16 steps
// on as loaded, so one shuffle per row and kind serves both groups.
//
// Work split: one block per SM owns a contiguous run of row tiles, and its
// (tile, step) pairs are cut into kMmaWarps equal contiguous ranges, one per
// warp, so every SM and every warp has the same number of groups to within
// one tile per block. A tile that lies inside one warp's range is written
// directly; a tile cut between warps leaves partial sums in shared memory,
// and the warp holding the tile's first step adds the later warps' partials
// in warp order, so the result does not depend on timing.

// Ring depth and warps per block (build-time tunables, defaults measured
// best), whether groups of 128 take this kernel (1) or the fp32 one above (0),
// and the layer size from which a single token takes it.
#ifndef AWQ_DECODE_MMA
#define AWQ_DECODE_MMA 1
#endif
#ifndef AWQ_MMA_STAGES
#define AWQ_MMA_STAGES 3
#endif
#ifndef AWQ_MMA_MIN_ONE_TOKEN_WEIGHTS
#define AWQ_MMA_MIN_ONE_TOKEN_WEIGHTS (int64_t(3) << 24)
#endif
#ifndef AWQ_MMA_WARPS
#define AWQ_MMA_WARPS 12
#endif
constexpr int kMmaWarps = AWQ_MMA_WARPS;
constexpr int kMmaThreads = kMmaWarps * 32;
constexpr int kMmaStages = AWQ_MMA_STAGES;  // pairs of groups per warp in the ring: kMmaStages - 1 in flight
constexpr int kMmaQStride = 20;             // staged words per (token, group, quarter): 16 + 4 of padding
constexpr int kMmaStageUnroll = 4;          // 16-byte loads of x in flight per thread while staging
constexpr int kMmaRingBytes = kMmaWarps * kMmaStages * 2 * 2 * 32 * 16;
constexpr int kMmaRedBytes = kMmaWarps * 2 * 4 * 32 * 4;  // per warp: a first and a last partial tile, 4 per lane

// Words per token region: 16 more than a multiple of 32, so two tokens read in one phase meet distinct banks.
__host__ __device__ constexpr int mma_token_words(int K) {
  return (K / 128) * 4 * kMmaQStride + (((K / 128) & 1) ? 0 : 16);
}
// Every accepted (n_tok, in) fits one block's shared memory (227 KB): the staged x of n_tok * in channels
// takes at most 2.5 bytes per channel plus 64 bytes per token.
static_assert(kMmaRingBytes + kMmaRedBytes + AWQ_W4A16_MAX_TOKEN_CHANNELS / 128 * 4 * kMmaQStride * 4 +
                      AWQ_W4A16_MAX_TOKENS * 16 * 4 <=
                  227 * 1024,
              "ring, partial sums and the largest staged x must fit one block's shared memory");

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The two constants of code_pair, held in registers for the kernel's life: with both as immediates the
// compiler spends a second integer instruction per pair.
struct PairConsts {
  uint32_t mask, bias;  // 0x000F000F, 0x43004300
  __device__ __forceinline__ PairConsts() {
    asm volatile("mov.b32 %0, 0x000F000F;" : "=r"(mask));
    asm volatile("mov.b32 %0, 0x43004300;" : "=r"(bias));
  }
};

// (128 + n, 128 + n') as a bf16 pair from a word whose nibbles n, n' sit at bits 0 and 16 (one
// three-input logic instruction: (ws & mask) | bias), minus the pair zz.
__device__ __forceinline__ uint32_t code_pair(uint32_t ws, uint32_t zz, const PairConsts& k) {
  uint32_t p;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(p) : "r"(ws), "r"(k.mask), "r"(k.bias));
  const __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&p),
                                   *reinterpret_cast<const __nv_bfloat162*>(&zz));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t bf16_pair_bits(float v) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(v, v);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Output rows ra, rb (= ra + 8) of tokens 2c, 2c + 1.
__device__ __forceinline__ void mma_store(float* __restrict__ y, int M, int N, int ra, int c, const float (&out)[4]) {
  const int rb = ra + 8, n0 = 2 * c, n1 = 2 * c + 1;
  if (ra < N && n0 < M && AWQ_IN((size_t)n0 * N + ra, 1, (size_t)M * N)) y[(size_t)n0 * N + ra] = out[0];
  if (ra < N && n1 < M && AWQ_IN((size_t)n1 * N + ra, 1, (size_t)M * N)) y[(size_t)n1 * N + ra] = out[1];
  if (rb < N && n0 < M && AWQ_IN((size_t)n0 * N + rb, 1, (size_t)M * N)) y[(size_t)n0 * N + rb] = out[2];
  if (rb < N && n1 < M && AWQ_IN((size_t)n1 * N + rb, 1, (size_t)M * N)) y[(size_t)n1 * N + rb] = out[3];
}

__global__ void __launch_bounds__(kMmaThreads, 1)
    w4a16_mma_kernel(const uint16_t* __restrict__ x, int M, int K, const int32_t* __restrict__ qweight,
                     const uint16_t* __restrict__ scales, const uint16_t* __restrict__ zeros, int N, float* __restrict__ y) {
  extern __shared__ uint4 mma_smem[];
  float* red = reinterpret_cast<float*>(mma_smem + kMmaRingBytes / 16);  // [warp][slot][4][32]
  // staged x: [token][group][quarter][20 words]
  uint32_t* xw = reinterpret_cast<uint32_t*>(mma_smem + (kMmaRingBytes + kMmaRedBytes) / 16);
  const int G = K >> 7;   // groups of 128 per row (even)
  const int P = G >> 1;   // steps per row: pairs of groups
  const int kw = K >> 3;  // code words per row
  const int tw = mma_token_words(K);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int quad = lane & ~3;
  const int tiles = (N + 15) >> 4;
  // this block's tiles, and this warp's steps within them (step = tile-major (tile, pair) index from t_lo)
  const int t_lo = (int)((int64_t)tiles * blockIdx.x / gridDim.x);
  const int t_hi = (int)((int64_t)tiles * (blockIdx.x + 1) / gridDim.x);
  const int64_t work = (int64_t)(t_hi - t_lo) * P;
  const int it_lo = (int)(work * warp / kMmaWarps), it_hi = (int)(work * (warp + 1) / kMmaWarps);
  const int first_tile = it_lo / P;  // block-relative
  const int first_p = it_lo - first_tile * P;

  // ring slot st: group 2p (uint4 [st * 128 + r * 32 + lane], r = 0 for row ra, 1 for rb), group 2p + 1 64 further
  uint4* ring = mma_smem + (size_t)warp * kMmaStages * 128 + lane;
  // lane c of a quad carries, for each group: c 0 the step of row ra, 1 of row rb, 2 the zero of ra, 3 of rb
  const uint16_t* sz_src = (c & 2) ? zeros : scales;
  uint32_t sz[kMmaStages];  // raw fp16 bits of the lane's step or zero for the pair's two groups, per ring slot
  // fetch state: the lane's code pieces of rows ra, rb and its steps or zeros, at the next pair to fetch
  const int32_t* fa = nullptr;
  const int32_t* fb = nullptr;
  const uint16_t* fs = nullptr;
  bool fva = false, fvb = false, fvo = false;
  int f_tile = first_tile, f_left = it_hi - it_lo, f_left_tile = P - first_p;
  auto aim = [&](int gi) {  // point the fetch state at group gi (even) of tile f_tile
    const int ra = (t_lo + f_tile) * 16 + g, rb = ra + 8, r_own = (c & 1) ? rb : ra;
    fva = ra < N && AWQ_IN((size_t)ra * kw + gi * 16 + 4 * c, 20, (size_t)N * kw);
    fvb = rb < N && AWQ_IN((size_t)rb * kw + gi * 16 + 4 * c, 20, (size_t)N * kw);
    fvo = r_own < N;
    fa = qweight + (size_t)(fva ? ra : 0) * kw + gi * 16 + 4 * c;
    fb = qweight + (size_t)(fvb ? rb : 0) * kw + gi * 16 + 4 * c;
    fs = sz_src + (size_t)(fvo ? r_own : 0) * G + gi;
  };
  aim(2 * first_p);
  // the next pair's codes into ring slot st and its two steps or zeros into sz[st]; nothing past the range
  auto fetch = [&](int st) {
    if (f_left > 0) {
      if (fva) {
        cp_async16(ring + st * 128, fa);
        cp_async16(ring + st * 128 + 64, fa + 16);
      }
      if (fvb) {
        cp_async16(ring + st * 128 + 32, fb);
        cp_async16(ring + st * 128 + 96, fb + 16);
      }
      uint32_t v = 0u;  // both groups' values in one aligned 32-bit load (row * G + gi is even)
      if (fvo && AWQ_IN((size_t)(fs - sz_src), 2, (size_t)N * G)) v = *reinterpret_cast<const uint32_t*>(fs);
      sz[st] = v;
      fa += 32;
      fb += 32;
      fs += 2;
      --f_left;
      if (--f_left_tile == 0 && f_left > 0) {
        ++f_tile;
        f_left_tile = P;
        aim(0);
      }
    }
    cp_async_commit();
  };
  // Programmatic dependent launch: the next kernel on the stream may start
  // launching now (its blocks take SMs as this kernel's leave). The codes,
  // steps and zeros of a packed layer are not written by the kernels before
  // this one, so the first pairs are fetched before waiting for them to
  // finish; x (the previous layer's output, in a decode step) and y are
  // touched only after. Without the launch attribute the wait returns at once.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the first pairs' codes are in flight while x is staged
#pragma unroll
  for (int st = 0; st < kMmaStages - 1; ++st) fetch(st);
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // stage x: chunk i (8 channels) of token n is (group gi, quarter c, chunk m) = (i / 16, i / 4 % 4, i % 4)
  {
    const int chunks = M * (K >> 3);
    const uint4* x4 = reinterpret_cast<const uint4*>(x);
    for (int base = threadIdx.x; base < chunks; base += kMmaThreads * kMmaStageUnroll) {
      uint4 v[kMmaStageUnroll];
#pragma unroll
      for (int u = 0; u < kMmaStageUnroll; ++u) {
        const int i = base + u * kMmaThreads;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (i < chunks && AWQ_IN((size_t)i * 8, 8, (size_t)M * K)) v[u] = x4[i];
      }
#pragma unroll
      for (int u = 0; u < kMmaStageUnroll; ++u) {
        const int i = base + u * kMmaThreads;
        if (i >= chunks) break;
        const int n = i / (K >> 3), r = i - n * (K >> 3);
        const int gi = r >> 4, cq = (r >> 2) & 3, m = r & 3;
        const uint4 w = make_uint4(__byte_perm(v[u].x, v[u].z, 0x5410), __byte_perm(v[u].x, v[u].z, 0x7632),
                                   __byte_perm(v[u].y, v[u].w, 0x5410), __byte_perm(v[u].y, v[u].w, 0x7632));
        *reinterpret_cast<uint4*>(xw + n * tw + (gi * 4 + cq) * kMmaQStride + 4 * m) = w;
      }
    }
  }
  __syncthreads();

  // MMA column g is token g; columns past the last token read token 0 (column j of the product depends on
  // column j of x only, and those columns are never stored)
  const uint32_t* xrow = xw + (size_t)(g < M ? g : 0) * tw + c * kMmaQStride;
  const PairConsts pk;
  float* red_mine = red + warp * 256 + lane;  // slot s, output i at [s * 128 + i * 32]
  float acc[4][4];
#pragma unroll
  for (int p = 0; p < 4; ++p)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[p][i] = 0.0f;
  // the tile's sums: to y (whole tile here) or to this warp's first or last slot
  auto flush = [&](int tile, bool whole) {
    float out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[i] = (acc[0][i] + acc[1][i]) + (acc[2][i] + acc[3][i]);
#pragma unroll
      for (int p = 0; p < 4; ++p) acc[p][i] = 0.0f;
    }
    if (whole) {
      mma_store(y, M, N, (t_lo + tile) * 16 + g, c, out);
    } else {
      float* slot = red_mine + (tile == first_tile ? 0 : 128);
#pragma unroll
      for (int i = 0; i < 4; ++i) slot[i * 32] = out[i];
    }
  };
  // 8 MMAs of one group of 16 rows: codes wa (row ra), wb (row rb), zero pairs zza, zzb, x at xg
  auto group_mma = [&](float (&d)[4], const uint4& qa, const uint4& qb, uint32_t zza, uint32_t zzb,
                       const uint32_t* xg) {
    const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
    const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint4 xv = *reinterpret_cast<const uint4*>(xg + 4 * m);  // b0, b1 of k-steps 2m and 2m + 1
      mma_bf16_16816(d, code_pair(wa[m], zza, pk), code_pair(wb[m], zzb, pk), code_pair(wa[m] >> 4, zza, pk),
                     code_pair(wb[m] >> 4, zzb, pk), xv.x, xv.y);
      mma_bf16_16816(d, code_pair(wa[m] >> 8, zza, pk), code_pair(wb[m] >> 8, zzb, pk),
                     code_pair(wa[m] >> 12, zza, pk), code_pair(wb[m] >> 12, zzb, pk), xv.z, xv.w);
    }
  };
  // the constant -256 k of each row against one group's activations (zero points outside [-128, 127])
  auto far_zero_mma = [&](float (&d)[4], float kf, const uint32_t* xg) {
    const float kfa = __shfl_sync(0xffffffffu, kf, quad + 2), kfb = __shfl_sync(0xffffffffu, kf, quad + 3);
    const uint32_t ka = bf16_pair_bits(-256.0f * kfa), kb2 = bf16_pair_bits(-256.0f * kfb);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint4 xv = *reinterpret_cast<const uint4*>(xg + 4 * m);
      mma_bf16_16816(d, ka, kb2, ka, kb2, xv.x, xv.y);
      mma_bf16_16816(d, ka, kb2, ka, kb2, xv.z, xv.w);
    }
  };
  // one pair of groups: codes from ring slot st, this lane's two steps or zeros from sz[st]
  int c_tile = first_tile, c_p = first_p;
  auto step = [&](int st) {
    cp_async_wait<kMmaStages - 2>();  // this pair's codes have landed (this thread's copies)
    const uint4 qa0 = ring[st * 128], qb0 = ring[st * 128 + 32];
    const uint4 qa1 = ring[st * 128 + 64], qb1 = ring[st * 128 + 96];
    const uint32_t own = sz[st];  // fp16 bits: group 2p low, 2p + 1 high
    fetch((st + kMmaStages - 1) % kMmaStages);  // into the slot the previous pair used
    // A zero z = z_lo + 256 k (z_lo in [-128, 128]) enters the MMAs as the bf16 value 128 + z_lo, exact like
    // (q - z_lo); -256 k is exact in bf16 too. The zero lanes (c = 2, 3) pack both groups' 128 + z_lo into
    // one word, the step lanes pass their two fp16 steps on as loaded: one shuffle per row and kind.
    const float f0 = __half2float(__ushort_as_half((unsigned short)own));
    const float f1 = __half2float(__ushort_as_half((unsigned short)(own >> 16)));
    const float kf0 = rintf(f0 * (1.0f / 256.0f)), kf1 = rintf(f1 * (1.0f / 256.0f));
    const __nv_bfloat162 zp = __floats2bfloat162_rn(128.0f + (f0 - 256.0f * kf0), 128.0f + (f1 - 256.0f * kf1));
    const uint32_t mine = (c & 2) ? *reinterpret_cast<const uint32_t*>(&zp) : own;
    const uint32_t sa = __shfl_sync(0xffffffffu, mine, quad), sb = __shfl_sync(0xffffffffu, mine, quad + 1);
    const uint32_t za = __shfl_sync(0xffffffffu, mine, quad + 2), zb = __shfl_sync(0xffffffffu, mine, quad + 3);
    const float sfa0 = __half2float(__ushort_as_half((unsigned short)sa));
    const float sfa1 = __half2float(__ushort_as_half((unsigned short)(sa >> 16)));
    const float sfb0 = __half2float(__ushort_as_half((unsigned short)sb));
    const float sfb1 = __half2float(__ushort_as_half((unsigned short)(sb >> 16)));
    const uint32_t zza0 = __byte_perm(za, 0u, 0x1010), zza1 = __byte_perm(za, 0u, 0x3232);  // (v, v) pairs
    const uint32_t zzb0 = __byte_perm(zb, 0u, 0x1010), zzb1 = __byte_perm(zb, 0u, 0x3232);
    const uint32_t* xg0 = xrow + (2 * c_p) * (4 * kMmaQStride);
    const uint32_t* xg1 = xg0 + 4 * kMmaQStride;
    float d0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, d1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    group_mma(d0, qa0, qb0, zza0, zzb0, xg0);
    group_mma(d1, qa1, qb1, zza1, zzb1, xg1);
    if (__any_sync(0xffffffffu, (c & 2) && (kf0 != 0.0f || kf1 != 0.0f))) {
      far_zero_mma(d0, kf0, xg0);
      far_zero_mma(d1, kf1, xg1);
    }
    float (&a0)[4] = acc[(2 * st) & 3];
    float (&a1)[4] = acc[(2 * st + 1) & 3];
    a0[0] = fmaf(sfa0, d0[0], a0[0]);
    a0[1] = fmaf(sfa0, d0[1], a0[1]);
    a0[2] = fmaf(sfb0, d0[2], a0[2]);
    a0[3] = fmaf(sfb0, d0[3], a0[3]);
    a1[0] = fmaf(sfa1, d1[0], a1[0]);
    a1[1] = fmaf(sfa1, d1[1], a1[1]);
    a1[2] = fmaf(sfb1, d1[2], a1[2]);
    a1[3] = fmaf(sfb1, d1[3], a1[3]);
    if (++c_p == P) {  // the tile's last pair: whole if this warp also had its first
      flush(c_tile, c_tile != first_tile || first_p == 0);
      c_p = 0;
      ++c_tile;
    }
  };
  int it = it_lo;
#pragma unroll 1
  for (; it + kMmaStages <= it_hi; it += kMmaStages) {
#pragma unroll
    for (int st = 0; st < kMmaStages; ++st) step(st);
  }
#pragma unroll
  for (int st = 0; st < kMmaStages - 1; ++st)
    if (it + st < it_hi) step(st);
  if (c_p != 0) flush(c_tile, false);  // the range ends inside a tile
  cp_async_wait<0>();
  __syncthreads();
  // a tile cut between warps: the warp holding its first pair adds the later warps' first-slot partials
  if (it_hi > it_lo && it_hi % P != 0) {
    const int lt = it_hi / P;  // this warp's last tile, continued by later warps
    if (lt * P >= it_lo) {
      float out[4];
      const float* own_slot = red_mine + (lt == first_tile ? 0 : 128);
#pragma unroll
      for (int i = 0; i < 4; ++i) out[i] = own_slot[i * 32];
      for (int w2 = warp + 1; w2 < kMmaWarps; ++w2) {
        const int lo2 = (int)(work * w2 / kMmaWarps), hi2 = (int)(work * (w2 + 1) / kMmaWarps);
        if (lo2 >= (lt + 1) * P) break;
        if (hi2 == lo2) continue;
#pragma unroll
        for (int i = 0; i < 4; ++i) out[i] += red[w2 * 256 + i * 32 + lane];
      }
      mma_store(y, M, N, (t_lo + lt) * 16 + g, c, out);
    }
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
  // groups of 128 with an even number of groups per row and 4-byte aligned steps and zeros: the
  // tensor-core product (it steps by pairs of groups, reading both groups' step or zero in one load), except
  // one token on a small layer, where the fp32 kernel's shorter start wins (measured)
  const bool pairs_ok = (K / 128) % 2 == 0 && (reinterpret_cast<uintptr_t>(scales) & 3u) == 0 &&
                        (reinterpret_cast<uintptr_t>(zeros) & 3u) == 0;
  if (AWQ_DECODE_MMA && group == 128 && pairs_ok && M >= 1 && M <= 8 &&
      (M >= 2 || N * K >= AWQ_MMA_MIN_ONE_TOKEN_WEIGHTS)) {
    int sms = 0;
    cudaError_t e = sm_count(&sms);
    if (e != cudaSuccess) return e;
    const int smem = kMmaRingBytes + kMmaRedBytes + (int)(M * mma_token_words((int)K) * 4);
    e = ensure_dynamic_smem((const void*)w4a16_mma_kernel, smem);
    if (e != cudaSuccess) return e;
    // one block per SM, each with a contiguous run of row tiles
    const int64_t tiles = (N + 15) / 16;
    const int64_t grid = tiles < (int64_t)sms ? tiles : (int64_t)sms;
    // launched so that it may overlap the previous kernel's tail (the kernel
    // waits for that kernel before it reads x)
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.gridDim = dim3((unsigned)grid);
    lc.blockDim = dim3(kMmaThreads);
    lc.dynamicSmemBytes = smem;
    lc.stream = st;
    lc.attrs = attr;
    lc.numAttrs = 1;
    e = cudaLaunchKernelEx(&lc, w4a16_mma_kernel, x, (int)M, (int)K, qweight, scales, zeros, (int)N, y);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
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
