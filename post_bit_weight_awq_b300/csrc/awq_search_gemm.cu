// Search product of the AWQ alpha grid on the 5th-generation tensor cores.
//
// For every alpha_i the search_scale listing of "AWQ: How Activation-Aware
// Quantization Saves 4-bit LLMs" needs the mean of (X W_hat_i^T - X W^T)^2.
// This kernel produces, per 128 x 256 output tile, the sum of those squares
// without writing the product to memory:
//
//   RESIDUAL form:  D = X (W_hat_i - W)^T  (operand slot i = bf16(W_hat_i - W))
//                   partial = sum D^2
//   REFERENCE form: Y = X W^T is computed once per output tile into tensor
//                   memory and stays resident; for each alpha, D_i = X W_hat_i^T
//                   and partial_i = sum (D_i - Y)^2.
//
// Structure of the single-CTA form (one CTA per SM, persistent over tiles,
// 192 threads; used for the REFERENCE form and the bounded-wait test aid):
//   warp 0, lane 0 : TMA producer. X tile [128 x 64] and operand tile
//                    [256 x 64] per stage, 128-byte swizzle, 4-stage ring.
//   warp 1         : allocates 512 tensor-memory columns; lane 0 issues
//                    tcgen05.mma (M=128, N=256, K=16, bf16 -> fp32) and
//                    commits completions to mbarriers.
//   warps 2..5     : epilogue. Each warp owns one 32-lane quarter of the
//                    accumulator (= 32 tokens), reads it with tcgen05.ld,
//                    squares and sums, and writes one fp32 per quarter.
// Tensor memory: two 256-column fp32 accumulators. RESIDUAL double-buffers
// them so the epilogue of a tile overlaps the next tile's MMAs; REFERENCE
// keeps Y in the second and accumulates X W_hat_i^T in the first.
// The default RESIDUAL product is the CTA-pair form further down.
// Every wait is bounded (wall time and iteration count): on a timeout the
// kernel records AWQ_ERR_TIMEOUT, stops all roles, lets its in-flight copies
// and MMAs land, frees tensor memory and returns.
#include "awq_device.cuh"
#include "awq_launch.h"
#include "awq_quant.cuh"

namespace awq {
namespace {

constexpr int BM = kTileM, BN = kTileN, BK = kTileK;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KiB
constexpr int B_BYTES = BN * BK * 2;  // 32 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;
// Token tiles per raster band (build-time tunables): the CTA-pair kernels
// (burst-length searches) and the single-CTA kernel (searches long enough to
// run at the power limit, where every DRAM byte costs energy).
#ifndef AWQ_RASTER_TILES_PAIR
#define AWQ_RASTER_TILES_PAIR 16
#endif
#ifndef AWQ_RASTER_TILES_SINGLE
#define AWQ_RASTER_TILES_SINGLE 16
#endif
constexpr int kRasterTokenTilesPair = AWQ_RASTER_TILES_PAIR;
constexpr int kRasterTokenTilesSingle = AWQ_RASTER_TILES_SINGLE;
constexpr int NUM_THREADS = 192;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + BAR_BYTES;
constexpr uint32_t IDESC = umma_idesc_bf16_f32(BM, BN);

struct Params {
  int mt, nt;         // token tiles, output-row tiles
  int kb;             // K blocks of 64
  int G;              // alphas
  int mtg;            // token-tile groups: ceil(mt / 2) for the CTA-pair form, mt for the single-CTA form
  int items;          // work items (RESIDUAL: G*mtg*nt; REFERENCE: mt*nt)
  int raster_group;   // tiles of the stationary operand per raster sweep
  int raster_n;       // 1: operand tiles stay, token tiles sweep; 0: the reverse
  uint64_t timeout_ns;
  float* partials;    // [G][mt][nt][4]
  uint32_t* status;
  float* dump;        // optional raw products [G][n_tok][N] (RESIDUAL): the W4A16 product's output, and a test aid
  double* row_acc;    // optional per-output-row sums of squared errors [G][N] (added to; nullptr: off)
  int n_tok, N;
  int withhold_first_fill;  // test aid: leave out each CTA's first operand fill
  // fused fake-quant (pair kernel with quantiser warps)
  const void* W;            // [N][K] bf16 bits or fp32
  int w_bf16;
  int K;
  int nstrips;              // 512-channel strips of K
  const float* s;           // [G][K]
  const float* inv_s;       // [G][K]
  uint16_t* op;             // [G][N][K] bf16, written by the quantiser warps
  uint32_t* ready;          // [G][nt] quantiser-warp arrivals per operand tile, then [G] per alpha,
                            // then the search progress word (see quantise_units)
  float qmax, floor_;
  int symmetric;            // zero point off (fixed z = 2^(b-1))
  int skip_unit;            // test aid: quantiser unit never written or published (-1: none)
};

// Tile t of an m_tiles x nt grid in raster order. Tiles are taken in bands
// of `group` tiles of the stationary operand (operand-row tiles if raster_n,
// else token tiles): within a band the other operand sweeps its whole range,
// so the band's panels of the stationary operand stay in L2 while each panel
// of the swept operand is read once per band.
// Raw products of one lane's token row, columns col0 .. col0 + 31 of alpha a,
// to dump[a][row][col]: 16-byte stores when the chunk is whole and rows are
// 16-byte aligned (N a multiple of 4), else one value at a time.
__device__ __forceinline__ void store_products(const Params& p, int a, int row, int col0, const uint32_t (&v)[32]) {
  const size_t base = ((size_t)a * p.n_tok + row) * p.N + col0;
  [[maybe_unused]] const size_t total = (size_t)p.G * p.n_tok * p.N;  // (bounds checks)
  if (col0 + 32 <= p.N && (p.N & 3) == 0) {
    if (!AWQ_IN(base, 32, total)) return;
    float4* d = reinterpret_cast<float4*>(p.dump + base);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      d[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]), __uint_as_float(v[4 * i + 2]),
                         __uint_as_float(v[4 * i + 3]));
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col0 + i < p.N && AWQ_IN(base + i, 1, total)) p.dump[base + i] = __uint_as_float(v[i]);
  }
}

// Per-column sums over the warp of the squares of 32 values per lane (lane =
// token row, value i = column i of a 32-column chunk): five exchange steps
// halve the columns each lane holds while summing over the lane pairs, so
// that lane l ends with column l summed over all 32 lanes (31 shuffles).
template <int N>
__device__ __forceinline__ void column_sum_step(float (&a)[32], int lane) {
  const bool upper = (lane & N) != 0;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float send = upper ? a[i] : a[i + N];
    const float keep = upper ? a[i + N] : a[i];
    a[i] = keep + __shfl_xor_sync(0xffffffffu, send, N);
  }
}

// Adds the warp's per-column sums of d^2 for the chunk's 32 columns to
// row_acc[alpha][col0 + lane] (columns past N are padding and are skipped).
__device__ __forceinline__ void add_row_sums(float (&sq)[32], int lane, double* row_acc, int alpha, int col0, int N,
                                             int G) {
  column_sum_step<16>(sq, lane);
  column_sum_step<8>(sq, lane);
  column_sum_step<4>(sq, lane);
  column_sum_step<2>(sq, lane);
  column_sum_step<1>(sq, lane);
  const int col = col0 + lane;
  if (col < N && AWQ_IN((size_t)alpha * N + col, 1, (size_t)G * N)) atomicAdd(&row_acc[(size_t)alpha * N + col], (double)sq[0]);
}

__device__ __forceinline__ void decode_tile(int t, int m_tiles, int nt, int group, int raster_n, int& mb, int& nb) {
  const int n_stat = raster_n ? nt : m_tiles;   // stationary dimension
  const int n_sweep = raster_n ? m_tiles : nt;  // swept dimension
  const int span = group * n_sweep;
  const int band = t / span;
  const int first = band * group;
  const int gsz = min(group, n_stat - first);
  const int r = t - band * span;
  const int i_stat = first + r % gsz;
  const int i_sweep = r / gsz;
  mb = raster_n ? i_sweep : i_stat;
  nb = raster_n ? i_stat : i_sweep;
}

template <bool REF>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    search_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                       const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (base_u32 & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* full = bars;               // [STAGES] TMA -> MMA
  uint64_t* empty = bars + STAGES;     // [STAGES] MMA -> TMA
  uint64_t* tfull = bars + 2 * STAGES; // [2] MMA -> epilogue
  uint64_t* tempty = tfull + 2;        // [2] epilogue -> MMA
  uint64_t* drain = tempty + 2;        // [1] final MMA completion
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int ncta = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int passes = REF ? p.G + 1 : 1;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t stage = 0, phase = 0;
      uint32_t used = 0, last_par = 0;  // per-stage bit: stage used; parity of its last fill
      bool ok = true;
      bool withhold = p.withhold_first_fill != 0;
      for (int it = cta; it < p.items && ok; it += ncta) {
        int a = 0, t = it;
        if (!REF) {
          a = it / (p.mtg * p.nt);
          t = it - a * p.mtg * p.nt;
        }
        int mg, nb;
        decode_tile(t, p.mtg, p.nt, p.raster_group, p.raster_n, mg, nb);
        const int mb = mg;
        for (int pass = 0; pass < passes && ok; ++pass) {
          const int slot = REF ? (pass == 0 ? p.G : pass - 1) : a;
          for (int kb = 0; kb < p.kb; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag, p.status)) {
              ok = false;
              break;
            }
            if (withhold) {
              // test aid: this stage is never filled, so the wait on it cannot complete
              withhold = false;
            } else {
              mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
              tma_load_2d(sA + stage * A_BYTES, &tmX, &full[stage], kb * BK, mb * BM);
              tma_load_3d(sB + stage * B_BYTES, &tmB, &full[stage], kb * BK, nb * BN, slot);
              used |= 1u << stage;
              last_par = (last_par & ~(1u << stage)) | (phase << stage);
            }
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Every copy issued must have landed before shared memory goes away.
      for (int s = 0; s < STAGES; ++s)
        if (used & (1u << s)) mbar_wait(&full[s], (last_par >> s) & 1u, p.timeout_ns, nullptr, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      uint32_t stage = 0, phase = 0;
      uint32_t ph = 0;  // bit b: parity of accumulator buffer b
      uint32_t local = 0;
      bool ok = true;
      for (int it = cta; it < p.items && ok; it += ncta, ++local) {
        for (int pass = 0; pass < passes && ok; ++pass) {
          // RESIDUAL: alternate buffers per tile. REFERENCE: Y -> buffer 1, D_i -> buffer 0.
          const int buf = REF ? (pass == 0 ? 1 : 0) : (int)(local & 1u);
          if (!mbar_wait(&tempty[buf], ((ph >> buf) & 1u) ^ 1u, p.timeout_ns, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
          for (int kb = 0; kb < p.kb; ++kb) {
            if (!mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t adesc = umma_desc_k_sw128(smem_u32(sA + stage * A_BYTES));
            const uint64_t bdesc = umma_desc_k_sw128(smem_u32(sB + stage * B_BYTES));
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              umma_bf16(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), IDESC,
                        (kb > 0 || k > 0) ? 1u : 0u);
            umma_commit(&empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit(&tfull[buf]);
          ph ^= 1u << buf;
        }
      }
      // Let every MMA issued finish before tensor memory is released.
      umma_commit(drain);
      mbar_wait(drain, 0u, p.timeout_ns, nullptr, p.status);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // tensor-memory lane quarter this warp may access
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t ph = 0;  // bit b: parity of accumulator buffer b
    uint32_t local = 0;
    bool ok = true;
    for (int it = cta; it < p.items && ok; it += ncta, ++local) {
      int a = 0, t = it;
      if (!REF) {
        a = it / (p.mtg * p.nt);
        t = it - a * p.mtg * p.nt;
      }
      int mg, nb;
      decode_tile(t, p.mtg, p.nt, p.raster_group, p.raster_n, mg, nb);
      const int mb = mg;
      if (REF) {
        // All lanes wait; the warp goes on only if every lane saw the phase
        // complete, so the warp-collective tensor-memory loads stay converged.
        if (!__all_sync(0xffffffffu, mbar_wait(&tfull[1], (ph >> 1) & 1u, p.timeout_ns, abort_flag, p.status)))
          break;
        tc_fence_after();
      }
      for (int pass = REF ? 1 : 0; pass < passes; ++pass) {
        const int buf = REF ? 0 : (int)(local & 1u);
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&tfull[buf], (ph >> buf) & 1u, p.timeout_ns, abort_flag, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc_addr = tmem_base + lane_base + (uint32_t)(buf * BN);
        float ss = 0.0f;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(acc_addr + (uint32_t)(c * 32), v);
          float sq[32];
          if (REF) {
            uint32_t y[32];
            tmem_ld_32x32b_x32(tmem_base + lane_base + (uint32_t)(BN + c * 32), y);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float d = __fsub_rn(__uint_as_float(v[i]), __uint_as_float(y[i]));
              ss = fmaf(d, d, ss);
              sq[i] = d * d;
            }
            if (p.row_acc != nullptr) add_row_sums(sq, lane, p.row_acc, pass - 1, nb * BN + c * 32, p.N, p.G);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float d = __uint_as_float(v[i]);
              ss = fmaf(d, d, ss);
              sq[i] = d * d;
            }
            if (p.row_acc != nullptr) add_row_sums(sq, lane, p.row_acc, a, nb * BN + c * 32, p.N, p.G);
            if (p.dump != nullptr) {
              const int row = mb * BM + q * 32 + lane;
              const int col0 = nb * BN + c * 32;
              if (row < p.n_tok) store_products(p, a, row, col0, v);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        ph ^= 1u << buf;
#pragma unroll
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const int alpha = REF ? pass - 1 : a;
        if (lane == 0 && mb < p.mt &&
            AWQ_IN((((size_t)alpha * p.mt + mb) * p.nt + nb) * 4 + q, 1, (size_t)p.G * p.mt * p.nt * 4))
          p.partials[((((size_t)alpha * p.mt + mb) * p.nt + nb) << 2) + q] = ss;
      }
      if (REF && ok) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[1]);
        ph ^= 2u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- CTA-pair form
//
// RESIDUAL form on CTA pairs (cta_group::2), the default search product.
// A cluster of two CTAs on neighbouring SMs computes 256 x 256 output tiles
// (two token tiles of 128 against one operand tile of 256 rows): each CTA
// loads its 128 token rows of X and its half (128 rows) of the operand tile
// into its own shared memory, and one thread of the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16), which reads A and B
// from both CTAs and accumulates each CTA's 128 rows in that CTA's tensor
// memory. Per stage each SM therefore receives 32 KiB for a 128 x 256 x 64
// product (48 KiB in the single-CTA form), so the ring holds kPairStages
// stages in the same shared memory.
//   full[s]   (even CTA) : both CTAs' copies of stage s landed (64 KiB);
//                          the odd CTA's copies report to it across the pair
//   empty[s]  (each CTA) : the pair's MMAs released stage s (commit multicast)
//   tfull[b]  (each CTA) : accumulator b is complete (commit multicast)
//   tempty[b] (even CTA) : all 8 epilogue warps of the pair read accumulator b
// Waits are bounded as in the single-CTA form; the final cluster barrier
// keeps each CTA alive until its peer no longer touches its shared memory or
// barriers.

constexpr int kPairStages = 6;
constexpr int kFqWarpsFused = 8;                                 // quantiser warps per CTA (fused form)
constexpr int kFusedThreads = NUM_THREADS + 32 * kFqWarpsFused;  // 448
constexpr int kFqStrip = 512;                                    // channels per quantiser unit

// Wait until *ctr >= need (acquire at GPU scope), bounded like mbar_wait.
__device__ __forceinline__ bool wait_counter(const uint32_t* ctr, uint32_t need, uint64_t timeout_ns,
                                             volatile int* abort_flag, uint32_t* status) {
  if (ld_acquire_gpu(ctr) >= need) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    __nanosleep(128);
    if (ld_acquire_gpu(ctr) >= need) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns) break;
    }
  }
  set_status(status, AWQ_ERR_TIMEOUT);
  *abort_flag = 1;
  return false;
}

// The lane's 16 scales and reciprocals, held in registers for a unit.
struct RegLane {
  const float2 (&s)[8];
  const float2 (&inv)[8];
  __device__ __forceinline__ void load_s(float2 (&v)[8]) const {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = s[i];
  }
  __device__ __forceinline__ void load_inv(float2 (&v)[8]) const {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = inv[i];
  }
};

__device__ __forceinline__ void ldg_lane16(const float* p, float2 (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  const float4 c = *reinterpret_cast<const float4*>(p + 64);
  const float4 d = *reinterpret_cast<const float4*>(p + 68);
  v[0] = make_float2(a.x, a.y);
  v[1] = make_float2(a.z, a.w);
  v[2] = make_float2(b.x, b.y);
  v[3] = make_float2(b.z, b.w);
  v[4] = make_float2(c.x, c.y);
  v[5] = make_float2(c.z, c.w);
  v[6] = make_float2(d.x, d.y);
  v[7] = make_float2(d.z, d.w);
}

// 16 weights of a lane: channels [c, c+8) and [c+64, c+72) of a row.
__device__ __forceinline__ void ldg_w16(const void* W, int w_bf16, size_t off, float2 (&w)[8]) {
  if (w_bf16) {
    const uint16_t* p = static_cast<const uint16_t*>(W) + off;
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    const uint4 b = *reinterpret_cast<const uint4*>(p + 64);
    const uint32_t x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = make_float2(bf16_lo(x[i]), bf16_hi(x[i]));
  } else {
    ldg_lane16(static_cast<const float*>(W) + off, w);
  }
}

// Quantiser warps of the fused form. The search operand of alpha a is cut
// into units (a, operand-row tile nb, 512-channel strip), numbered a-major
// then nb then strip, i.e. in the order the search consumes them, and dealt
// to the CTAs round-robin. The CTA's 8 quantiser warps take 32 rows of the
// unit's 256 each (lane layout and arithmetic as in the fake-quant kernel,
// with the lane's scales held in registers for the unit), then each warp
// publishes its rows: every lane fences (generic -> async proxy, then GPU
// scope), and lane 0 adds 1 to ready[a][nb] and to the alpha's counter with
// release semantics. A tile is complete when its counter reaches
// nstrips * 8, an alpha when its counter reaches nt * nstrips * 8. The
// quantisers never wait, so every unit is finished as long as all CTAs of
// the launch are resident, which the grid size ensures on a GPU that runs
// nothing else. (Holding the quantisers a fixed number of alphas ahead of
// the products, so that each operand is written just before it is read,
// measured no faster on the benchmark layers.)
template <int GROUP>
__device__ __forceinline__ void quantise_units(const Params& p, int fw, int lane) {
  const int grp = lane >> 3, sub = lane & 7;
  const QuantSpec qs = make_quant_spec(p.qmax, p.floor_, p.symmetric != 0);
  const int per_a = p.nt * p.nstrips;
  const int units = p.G * per_a;
  const size_t slot = (size_t)p.N * p.K;
  uint32_t* ready_alpha = p.ready + (size_t)p.G * p.nt;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    if (u == p.skip_unit) continue;  // test aid: the tile of this unit never becomes ready
    const int a = u / per_a;
    const int rem = u - a * per_a;
    const int nb = rem / p.nstrips;
    const int col0 = (rem - nb * p.nstrips) * kFqStrip;
    const int ncols = min(kFqStrip, p.K - col0);
    const bool active = grp * 128 < ncols;  // groups past a partial strip repeat group 0, store nothing
    const int c = col0 + (active ? grp * 128 : 0) + sub * 8;
    const int r0 = nb * BN + fw * 32;
    const int r1 = min(r0 + 32, p.N);
    if (r0 < r1) {
      float2 sv[8] = {}, iv[8] = {};
      if (AWQ_IN((size_t)a * p.K + c, 72, (size_t)p.G * p.K)) {
        ldg_lane16(p.s + (size_t)a * p.K + c, sv);
        ldg_lane16(p.inv_s + (size_t)a * p.K + c, iv);
      }
      [[maybe_unused]] const size_t wn_elems = (size_t)p.N * p.K;  // (bounds checks)
      float2 wn[8] = {};
      if (AWQ_IN((size_t)r0 * p.K + c, 72, wn_elems)) ldg_w16(p.W, p.w_bf16, (size_t)r0 * p.K + c, wn);
      for (int r = r0; r < r1; ++r) {
        float2 w[8], nw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          w[i] = wn[i];
          nw[i] = make_float2(-w[i].x, -w[i].y);
        }
        if (r + 1 < r1 && AWQ_IN((size_t)(r + 1) * p.K + c, 72, wn_elems))
          ldg_w16(p.W, p.w_bf16, (size_t)(r + 1) * p.K + c, wn);
        uint32_t o[8];
        fq_lane16<false, GROUP>(w, nw, RegLane{sv, iv}, qs, o);
        if (active && AWQ_IN((size_t)a * slot + (size_t)r * p.K + c, 72, (size_t)p.G * slot)) {
          uint4* dst = reinterpret_cast<uint4*>(p.op + (size_t)a * slot + (size_t)r * p.K + c);
          dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
          dst[8] = make_uint4(o[4], o[5], o[6], o[7]);  // 64 channels further on
        }
      }
    }
    fence_proxy_async_global();
    __threadfence();
    __syncwarp();
    if (lane == 0) {
      if (AWQ_IN((size_t)a * p.nt + nb, 1, (size_t)p.G * p.nt)) red_release_gpu_add(&p.ready[(size_t)a * p.nt + nb], 1u);
      if (AWQ_IN(a, 1, p.G)) red_release_gpu_add(&ready_alpha[a], 1u);
    }
  }
}
constexpr int PA_BYTES = BM * BK * 2;          // 16 KiB: this CTA's token rows
constexpr int PB_BYTES = (BN / 2) * BK * 2;    // 16 KiB: this CTA's half of the operand rows
constexpr int PSTAGE_BYTES = PA_BYTES + PB_BYTES;
constexpr int PAIR_SMEM_BYTES = kPairStages * PSTAGE_BYTES + 1024 + BAR_BYTES;
constexpr uint32_t PAIR_IDESC = umma_idesc_bf16_f32(2 * BM, BN);
static_assert(PAIR_SMEM_BYTES <= 232448, "shared memory per CTA");

template <bool FUSED, int GROUP = 128>
__global__ void __launch_bounds__(FUSED ? kFusedThreads : NUM_THREADS, 1)
    search_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                            const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (base_u32 & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kPairStages * PA_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kPairStages * PB_BYTES);
  uint64_t* full = bars;                     // [kPairStages]
  uint64_t* empty = bars + kPairStages;      // [kPairStages]
  uint64_t* tfull = bars + 2 * kPairStages;  // [2]
  uint64_t* tempty = tfull + 2;              // [2]
  uint64_t* drain = tempty + 2;              // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank() & 1u;
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  constexpr uint16_t kPairMask = 3;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 8);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the even CTA's barriers exist before its peer reports to them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer (both CTAs)
      uint32_t stage = 0, phase = 0;
      uint32_t used = 0, last_par = 0;
      bool ok = true;
      int started = -1, verified = -1;  // fused form: newest alpha started / known fully quantised
      for (int it = pair; it < p.items && ok; it += npairs) {
        const int a = it / (p.mtg * p.nt);
        const int t = it - a * p.mtg * p.nt;
        int mg, nb;
        decode_tile(t, p.mtg, p.nt, p.raster_group, p.raster_n, mg, nb);
        const int mb = mg * 2 + (int)rank;
        if (FUSED) {
          if (a > started) {
            started = a;
            atomicMax(p.ready + (size_t)p.G * p.nt + p.G, (uint32_t)(a + 1));  // progress word (diagnostic)
          }
          if (a != verified) {
            // the quantiser warps of every CTA have written this operand tile
            // (or the whole alpha, after which no further check is needed)
            const uint32_t* alpha_ctr = p.ready + (size_t)p.G * p.nt + a;
            if (ld_acquire_gpu(alpha_ctr) >= (uint32_t)(p.nt * p.nstrips * kFqWarpsFused)) {
              verified = a;
            } else if (!wait_counter(&p.ready[(size_t)a * p.nt + nb], (uint32_t)(p.nstrips * kFqWarpsFused),
                                     p.timeout_ns, abort_flag, p.status)) {
              ok = false;
              break;
            }
            fence_proxy_async_global();  // order the TMA reads after the quantisers' generic-proxy writes
          }
        }
        for (int kb = 0; kb < p.kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t fbar = mapa_shared(&full[stage], 0);
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * PSTAGE_BYTES);
          tma_load_2d_pair(sA + stage * PA_BYTES, &tmX, fbar, kb * BK, mb * BM);
          tma_load_3d_pair(sB + stage * PB_BYTES, &tmB, fbar, kb * BK, nb * BN + (int)rank * (BN / 2), a);
          used |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every copy issued by the pair reports to the even CTA's barriers: it
      // waits for all of them before the final cluster barrier.
      if (leader)
        for (int s = 0; s < kPairStages; ++s)
          if (used & (1u << s)) mbar_wait(&full[s], (last_par >> s) & 1u, p.timeout_ns, nullptr, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ MMA issuer (even CTA)
      uint32_t stage = 0, phase = 0;
      uint32_t ph = 0;
      uint32_t local = 0;
      bool ok = true;
      for (int it = pair; it < p.items && ok; it += npairs, ++local) {
        const int buf = (int)(local & 1u);
        if (!mbar_wait(&tempty[buf], ((ph >> buf) & 1u) ^ 1u, p.timeout_ns, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
        for (int kb = 0; kb < p.kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = umma_desc_k_sw128(smem_u32(sA + stage * PA_BYTES));
          const uint64_t bdesc = umma_desc_k_sw128(smem_u32(sB + stage * PB_BYTES));
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16_pair(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), PAIR_IDESC,
                           (kb > 0 || k > 0) ? 1u : 0u);
          umma_commit_pair_multicast(&empty[stage], kPairMask);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_multicast(&tfull[buf], kPairMask);
        ph ^= 1u << buf;
      }
      umma_commit_pair(drain);
      mbar_wait(drain, 0u, p.timeout_ns, nullptr, p.status);
    }
  } else if (warp < 6) {
    // -------------------------------------------------------------- epilogue (both CTAs)
    const int q = warp & 3;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t ph = 0;
    uint32_t local = 0;
    for (int it = pair; it < p.items; it += npairs, ++local) {
      const int a = it / (p.mtg * p.nt);
      const int t = it - a * p.mtg * p.nt;
      int mg, nb;
      decode_tile(t, p.mtg, p.nt, p.raster_group, p.raster_n, mg, nb);
      const int mb = mg * 2 + (int)rank;
      const int buf = (int)(local & 1u);
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[buf], (ph >> buf) & 1u, p.timeout_ns, abort_flag, p.status)))
        break;
      tc_fence_after();
      const uint32_t acc_addr = tmem_base + lane_base + (uint32_t)(buf * BN);
      float ss = 0.0f;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(acc_addr + (uint32_t)(c * 32), v);
        float sq[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float d = __uint_as_float(v[i]);
          ss = fmaf(d, d, ss);
          sq[i] = d * d;
        }
        if (p.row_acc != nullptr) add_row_sums(sq, lane, p.row_acc, a, nb * BN + c * 32, p.N, p.G);
        if (p.dump != nullptr) {
          const int row = mb * BM + q * 32 + lane;
          const int col0 = nb * BN + c * 32;
          if (row < p.n_tok) store_products(p, a, row, col0, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(&tempty[buf], 0));
      ph ^= 1u << buf;
#pragma unroll
      for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0 && mb < p.mt &&
          AWQ_IN((((size_t)a * p.mt + mb) * p.nt + nb) * 4 + q, 1, (size_t)p.G * p.mt * p.nt * 4))
        p.partials[((((size_t)a * p.mt + mb) * p.nt + nb) << 2) + q] = ss;
    }
  } else if (FUSED) {
    // -------------------------------------------------------------- quantiser warps (both CTAs)
    quantise_units<GROUP>(p, warp - 6, lane);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer no longer copies into, reports to or arrives on this CTA
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

// Single-CTA launch: one persistent CTA per SM (fewer if there are fewer items).
template <bool REF>
cudaError_t launch_single(const CUtensorMap& tmX, const CUtensorMap& tmB, const Params& p, int sms, cudaStream_t st) {
  cudaError_t e = ensure_dynamic_smem((const void*)search_gemm_kernel<REF>, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int grid = p.items < sms ? p.items : sms;
  search_gemm_kernel<REF><<<grid, NUM_THREADS, SMEM_BYTES, st>>>(tmX, tmB, p);
  return cudaGetLastError();
}

template <bool FUSED, int GROUP = 128>
cudaError_t launch_pair(const CUtensorMap& tmX, const CUtensorMap& tmB, const Params& p, int sms, cudaStream_t st) {
  constexpr int threads = FUSED ? kFusedThreads : NUM_THREADS;
  cudaError_t e = ensure_dynamic_smem((const void*)search_gemm_pair_kernel<FUSED, GROUP>, PAIR_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.blockDim = dim3(threads);
  lc.dynamicSmemBytes = PAIR_SMEM_BYTES;
  lc.stream = st;
  lc.attrs = attr;
  lc.numAttrs = 1;
  int pairs = sms / 2;
  lc.gridDim = dim3(2 * pairs);
  int active = 0;
  e = cudaOccupancyMaxActiveClusters(&active, search_gemm_pair_kernel<FUSED, GROUP>, &lc);
  if (e != cudaSuccess) return e;
  if (active > 0 && active < pairs) pairs = active;
  // The fused form keeps every pair even without search items of its own:
  // its quantiser warps serve the operand tiles of other pairs.
  if (!FUSED && pairs > p.items) pairs = p.items;
  lc.gridDim = dim3(2 * pairs);
  return cudaLaunchKernelEx(&lc, search_gemm_pair_kernel<FUSED, GROUP>, tmX, tmB, p);
}

// Tensor maps and tiling of a search launch. CM: CTAs that split one 256-row
// operand tile (2 for the CTA-pair kernels, each loading its 128-row half;
// 1 for the single-CTA kernel).
cudaError_t setup_search(const uint16_t* X, int64_t n_tok, int64_t K, const uint16_t* op, int64_t N,
                         const awq_config& cfg, int CM, CUtensorMap* tmX, CUtensorMap* tmB, Params* pp, int* sms) {
  const bool ref = cfg.loss_form == AWQ_LOSS_REFERENCE;
  const int G = cfg.n_grid;
  const int slots = ref ? G + 1 : G;
  const cuuint64_t xd[2] = {(cuuint64_t)K, (cuuint64_t)n_tok};
  const cuuint32_t xb[2] = {(cuuint32_t)BK, (cuuint32_t)BM};
  const cuuint64_t bd[3] = {(cuuint64_t)K, (cuuint64_t)N, (cuuint64_t)slots};
  const cuuint32_t bb[3] = {(cuuint32_t)BK, (cuuint32_t)(BN / CM), 1u};
  if (!make_map(tmX, X, 2, xd, xb) || !make_map(tmB, op, 3, bd, bb)) return cudaErrorInvalidValue;

  cudaError_t e = sm_count(sms);
  if (e != cudaSuccess) return e;

  Params p = {};
  p.mt = (int)((n_tok + BM - 1) / BM);
  p.nt = (int)((N + BN - 1) / BN);
  p.mtg = (p.mt + CM - 1) / CM;
  p.kb = (int)(K / BK);
  p.G = G;
  p.items = ref ? p.mt * p.nt : G * p.mtg * p.nt;
  // L2 raster: bands of token tiles stay in L2 while the operand tiles sweep
  // past them, so each operand tile is read from DRAM once per band.
  p.raster_n = 0;
  const int band = CM == 2 ? kRasterTokenTilesPair : kRasterTokenTilesSingle;
  p.raster_group = (band + CM - 1) / CM;
  if (p.raster_group > p.mtg) p.raster_group = p.mtg;
  const uint32_t ms = cfg.wait_timeout_ms ? cfg.wait_timeout_ms : 2000u;
  p.timeout_ns = (uint64_t)ms * 1000000ull;
  p.n_tok = (int)n_tok;
  p.N = (int)N;
  p.K = (int)K;
  p.skip_unit = -1;
  *pp = p;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_search_gemm(const uint16_t* X, int64_t n_tok, int64_t K, const uint16_t* op, int64_t N,
                               const awq_config& cfg, float* partials, uint32_t* status, cudaStream_t st,
                               float* dump, int withhold_first_fill, int single_cta, double* row_acc) {
  const bool ref = cfg.loss_form == AWQ_LOSS_REFERENCE;
  // the CTA-pair kernel for the RESIDUAL form; the single-CTA kernel for the
  // REFERENCE form, the withheld-fill test aid, or when asked for
  const bool pair = !ref && !withhold_first_fill && !single_cta;
  CUtensorMap tmX, tmB;
  Params p;
  int sms = 0;
  cudaError_t e = setup_search(X, n_tok, K, op, N, cfg, pair ? 2 : 1, &tmX, &tmB, &p, &sms);
  if (e != cudaSuccess) return e;
  p.partials = partials;
  p.status = status;
  p.dump = ref ? nullptr : dump;
  p.row_acc = row_acc;
  p.withhold_first_fill = withhold_first_fill;
  if (ref) e = launch_single<true>(tmX, tmB, p, sms, st);
  else if (pair) e = launch_pair<false>(tmX, tmB, p, sms, st);
  else e = launch_single<false>(tmX, tmB, p, sms, st);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_search_fused(const void* W, int w_dtype, const uint16_t* X, int64_t n_tok, int64_t K,
                                const float* s, const float* inv_s, int64_t N, const awq_config& cfg, uint16_t* op,
                                float* partials, uint32_t* ready, uint32_t* status, cudaStream_t st, float* dump,
                                int skip_unit, double* row_acc) {
  if (cfg.loss_form != AWQ_LOSS_RESIDUAL) return cudaErrorInvalidValue;
  CUtensorMap tmX, tmB;
  Params p;
  int sms = 0;
  cudaError_t e = setup_search(X, n_tok, K, op, N, cfg, 2, &tmX, &tmB, &p, &sms);
  if (e != cudaSuccess) return e;
  p.partials = partials;
  p.status = status;
  p.dump = dump;
  p.row_acc = row_acc;
  p.W = W;
  p.w_bf16 = w_dtype == AWQ_BF16 ? 1 : 0;
  p.nstrips = (int)((K + kFqStrip - 1) / kFqStrip);
  p.s = s;
  p.inv_s = inv_s;
  p.op = op;
  p.ready = ready;
  p.qmax = (float)((1 << cfg.w_bit) - 1);
  p.floor_ = cfg.delta_floor;
  p.symmetric = cfg.zero_point == 0 ? 1 : 0;
  p.skip_unit = skip_unit;
  e = cudaMemsetAsync(ready, 0, fused_ready_words(p.G, p.nt) * sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  switch (cfg.group) {
    case 32: e = launch_pair<true, 32>(tmX, tmB, p, sms, st); break;
    case 64: e = launch_pair<true, 64>(tmX, tmB, p, sms, st); break;
    case 128: e = launch_pair<true, 128>(tmX, tmB, p, sms, st); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

#ifdef AWQ_CHECKED
cudaError_t take_oob_search(unsigned long long* out) { return take_oob_record(out); }
#endif

}  // namespace awq
