// Gram form of the alpha search's loss on the 5th-generation tensor cores.
//
// The search_scale listing of "AWQ: How Activation-Aware Quantization Saves
// 4-bit LLMs" scores alpha_i by the mean over tokens t and output rows r of
// (X W_hat_i^T - X W^T)[t][r]^2. With D_i = W_hat_i - W (the RESIDUAL
// operand, bf16 [out][in]) and C = X^T X (in x in, symmetric):
//
//   sum_t sum_r (X D_i^T)[t][r]^2 = sum_r D_i[r] C D_i[r]^T,
//
// an exact identity. The direct product costs 2 n_tok out in flops per
// alpha; here C costs n_tok in^2 (the blocks on and below the diagonal) once
// and each alpha out in^2, because with column blocks of 256 channels,
// jb(x) = x / 256, only blocks on and below the diagonal are needed:
//
//   D C D^T = sum_c D[c] sum_{j: jb(j) <= jb(c)} H[c][j] D[j],
//   H[c][j] = C[c][j] * (2 if jb(j) < jb(c), 1 if jb(j) == jb(c)).
//
// That is fewer flops than the direct product whenever in < 2 n_tok.
//
// Kernels:
//   transpose_kernel : Xt [in][n_pad] = X^T, zero columns from n_tok to n_pad
//                      (n_tok rounded up to 64), so that both operands of
//                      Xt Xt^T are K-major for the tensor core.
//   gram_kernel<H>   : H as bf16 [in][in] (blocks on and below the diagonal
//                      only): 128 x 256 tiles of Xt Xt^T over all tokens,
//                      scaled (x2 or x1) and rounded to bf16 in the epilogue.
//   gram_kernel<LOSS>: for each alpha, 128 x 256 tiles of D_i H^T over the
//                      tile's prefix of column blocks; the epilogue adds
//                      P[r][c] * D_i[r][c] over the tile, so no product
//                      leaves the chip.
// Both gram_kernel forms have the single-CTA structure of the direct search
// product (one CTA per SM, persistent): warp 0 lane 0 feeds a 4-stage TMA
// ring (A tile 128 x 64, B tile 256 x 64, 128-byte swizzle), warp 1 owns
// 512 tensor-memory columns (two 256-column fp32 accumulators, so one
// tile's epilogue overlaps the next tile's MMAs) and lane 0 issues
// tcgen05.mma (M 128, N 256, K 16), warps 2..9 are the epilogue (warp w
// reads lanes 32 (w % 4) .. + 31 of the accumulator and one half of its
// columns, so that the chain of tensor-memory loads per warp is short).
// Every wait is bounded.
//
// Work of the loss kernel: the tile (alpha a, row block rb of 128 output
// rows, column block cb of 256 channels) costs 4 (cb + 1) k-blocks of 64
// (fewer for a last, half block). An item is row block rb with the column
// blocks cb and nC-1-cb, so every item costs 4 (nC + 1) k-blocks (an odd
// middle block is an item of its own). Items are dealt to the CTAs round
// robin in the order (alpha, group of kGramRowGroup row blocks, column-block
// pair, row block): neighbouring CTAs take the same pair for neighbouring
// rows, all CTAs start their items together and take equally long, so the
// CTAs of a group load the same tiles of H at the same time, which the L2
// serves as one stream instead of many. Each item writes one fp32 sum per
// epilogue warp: partials [n_grid][items per alpha][8]. The order of all
// sums is fixed by the shape, so the result does not depend on the GPU.
//
// Rounding: C is accumulated in fp32 over all tokens and rounded to bf16
// once (relative 2^-9 per entry, the x2 is exact). With the diagonal of C
// dominant that moves the loss by about 2^-9 / sqrt(in) relative; D_i has
// the bf16 rounding of the direct RESIDUAL product.
#include "awq_device.cuh"
#include "awq_launch.h"

namespace awq {
namespace {

constexpr int BM = kTileM, BN = kTileN, BK = kTileK;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KiB
constexpr int B_BYTES = BN * BK * 2;  // 32 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int EPI_WARPS = kGramEpilogueWarps;  // two per tensor-memory lane quarter
constexpr int EPI_COLS = BN * 4 / EPI_WARPS;   // accumulator columns per epilogue warp
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + BAR_BYTES;
constexpr uint32_t IDESC = umma_idesc_bf16_f32(BM, BN);
constexpr int KB_PER_COL_BLOCK = BN / BK;  // k-blocks of 64 in a 256-channel block

struct GramParams {
  int K;              // in
  int N;              // out (loss kernel)
  int G;              // alphas (loss kernel)
  // H kernel
  int kb_tok;         // k-blocks over tokens (n_pad / 64)
  int items;          // tiles on and below the block diagonal
  // loss kernel
  int nC;             // 256-channel column blocks: ceil(K / 256)
  int kbK;            // K / 64
  int nR;             // 128-row blocks of D_i: ceil(N / 128)
  int nP;             // column-block pairs: ceil(nC / 2)
  int per_alpha;      // items per alpha: nR * nP
  uint64_t timeout_ns;
  uint32_t* status;
  uint16_t* H;          // [K][K] bf16 (H kernel output)
  const uint16_t* op;   // [G][N][K] bf16 D_i (loss epilogue)
  float* partials;      // [G][nR * nP][EPI_WARPS]
  double* row_acc;      // optional [G][N], per-row sums added (loss kernel)
  int withhold_first_fill;  // test aid: leave out each CTA's first ring fill (loss kernel)
};

// ---------------------------------------------------------------- H tiles
//
// Tile i of the H kernel: 128-row tile ct of H and 256-column tile jt, with
// jt <= ct / 2 (on or below the block diagonal), in order of ct then jt.
// Tiles before ct = 2m + b number (m + 1)(m + b).
__device__ __forceinline__ void decode_h_tile(int i, int& ct, int& jt) {
  int m = (int)sqrtf((float)i);
  for (int g = 0; g < 8 && m > 0 && m * (m + 1) > i; ++g) --m;
  for (int g = 0; g < 8 && (m + 1) * (m + 2) <= i; ++g) ++m;
  if (i < (m + 1) * (m + 1)) {
    ct = 2 * m;
    jt = i - m * (m + 1);
  } else {
    ct = 2 * m + 1;
    jt = i - (m + 1) * (m + 1);
  }
}

// ---------------------------------------------------------------- loss items
//
// k-blocks of a tile in column block cb: the prefix of 256-channel blocks up
// to and including cb (a last, half block has 2 instead of 4).
__device__ __forceinline__ int tile_kblocks(const GramParams& p, int cb) {
  return min(KB_PER_COL_BLOCK * (cb + 1), p.kbK);
}

// Item t (< G * per_alpha) of the loss kernel: alpha a, row block rb and
// column-block pair pp (blocks pp and nC-1-pp). Within an alpha the row
// blocks go in groups of kGramRowGroup (the last group may be shorter), and
// within a group pair-major, row-minor.
__device__ __forceinline__ void decode_item(const GramParams& p, int t, int& a, int& rb, int& pp) {
  a = t / p.per_alpha;
  const int u = t - a * p.per_alpha;
  const int full = p.nR / kGramRowGroup;  // whole groups
  const int span = p.nP * kGramRowGroup;   // items of a whole group
  int g, local, rows;
  if (u < full * span) {
    g = u / span;
    local = u - g * span;
    rows = kGramRowGroup;
  } else {
    g = full;
    local = u - full * span;
    rows = p.nR - full * kGramRowGroup;
  }
  pp = local / rows;
  rb = g * kGramRowGroup + (local - pp * rows);
}

// The roles of both kernels walk the same sequence of pieces: fn(a, m_tile,
// n_tile, kb0, kb1, item_first, item_last, item) for every tile of every
// item this CTA takes. Returns false if fn does.
template <bool LOSS, typename Fn>
__device__ __forceinline__ bool for_each_piece(const GramParams& p, int cta, int ncta, Fn&& fn) {
  if constexpr (!LOSS) {
    for (int it = cta; it < p.items; it += ncta) {
      int ct, jt;
      decode_h_tile(it, ct, jt);
      if (!fn(0, ct, jt, 0, p.kb_tok, true, true, it)) return false;
    }
  } else {
    for (int it = cta; it < p.G * p.per_alpha; it += ncta) {
      int a, rb, pp;
      decode_item(p, it, a, rb, pp);
      const int cb2 = p.nC - 1 - pp;  // the long tile; the same block for an odd middle one
      if (!fn(a, rb, pp, 0, tile_kblocks(p, pp), true, cb2 == pp, it)) return false;
      if (cb2 != pp && !fn(a, rb, cb2, 0, tile_kblocks(p, cb2), false, true, it)) return false;
    }
  }
  return true;
}

__device__ __forceinline__ float dot_bf16x8(const float* v, uint4 d, float acc) {
  acc = fmaf(v[0], bf16_lo(d.x), acc);
  acc = fmaf(v[1], bf16_hi(d.x), acc);
  acc = fmaf(v[2], bf16_lo(d.y), acc);
  acc = fmaf(v[3], bf16_hi(d.y), acc);
  acc = fmaf(v[4], bf16_lo(d.z), acc);
  acc = fmaf(v[5], bf16_hi(d.z), acc);
  acc = fmaf(v[6], bf16_lo(d.w), acc);
  acc = fmaf(v[7], bf16_hi(d.w), acc);
  return acc;
}

template <bool LOSS>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gram_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GramParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (base_u32 & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* full = bars;                // [STAGES] TMA -> MMA
  uint64_t* empty = bars + STAGES;      // [STAGES] MMA -> TMA
  uint64_t* tfull = bars + 2 * STAGES;  // [2] MMA -> epilogue
  uint64_t* tempty = tfull + 2;         // [2] epilogue -> MMA
  uint64_t* drain = tempty + 2;         // [1] final MMA completion
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
      mbar_init(&tempty[b], EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
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

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t stage = 0, phase = 0;
      uint32_t used = 0, last_par = 0;  // per-stage bit: stage used; parity of its last fill
      bool withhold = p.withhold_first_fill != 0;
      for_each_piece<LOSS>(p, cta, ncta, [&](int a, int mt, int nt, int kb0, int kb1, bool, bool, int) {
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag, p.status)) return false;
          if (withhold) {
            // test aid: this stage is never filled, so the wait on it cannot complete
            withhold = false;
          } else {
            mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
            if constexpr (LOSS) {
              tma_load_3d(sA + stage * A_BYTES, &tmA, &full[stage], kb * BK, mt * BM, a);
            } else {
              tma_load_2d(sA + stage * A_BYTES, &tmA, &full[stage], kb * BK, mt * BM);
            }
            tma_load_2d(sB + stage * B_BYTES, &tmB, &full[stage], kb * BK, nt * BN);
            used |= 1u << stage;
            last_par = (last_par & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        return true;
      });
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
      for_each_piece<LOSS>(p, cta, ncta, [&](int, int, int, int kb0, int kb1, bool, bool, int) {
        if (kb0 == kb1) return true;  // an empty piece uses no accumulator
        const int buf = (int)(local & 1u);
        if (!mbar_wait(&tempty[buf], ((ph >> buf) & 1u) ^ 1u, p.timeout_ns, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.status)) return false;
          tc_fence_after();
          const uint64_t adesc = umma_desc_k_sw128(smem_u32(sA + stage * A_BYTES));
          const uint64_t bdesc = umma_desc_k_sw128(smem_u32(sB + stage * B_BYTES));
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), IDESC,
                      (kb > kb0 || k > 0) ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        umma_commit(&tfull[buf]);
        ph ^= 1u << buf;
        ++local;
        return true;
      });
      // Let every MMA issued finish before tensor memory is released.
      umma_commit(drain);
      mbar_wait(drain, 0u, p.timeout_ns, nullptr, p.status);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int ew = warp - 2;                         // epilogue warp 0 .. EPI_WARPS-1
    const int q = warp & 3;                          // tensor-memory lane quarter this warp may access
    const int col_base = (ew >> 2) * EPI_COLS;       // its half of the accumulator's columns
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t ph = 0;
    uint32_t local = 0;
    float item_sum = 0.0f;
    for_each_piece<LOSS>(p, cta, ncta, [&](int a, int mt, int nt, int kb0, int kb1, bool first, bool last, int flat) {
      if constexpr (LOSS) {
        if (first) item_sum = 0.0f;
      }
      if (kb0 < kb1) {
        const int buf = (int)(local & 1u);
        const int row = mt * BM + q * 32 + lane;  // LOSS: output row of D_i; H: row c of H
        if constexpr (LOSS) {
          // this lane's 128 values of D_i[row][nt * 256 + col_base ...], fetched while the MMAs run
          uint4 d[EPI_COLS / 8];
          const bool row_ok = row < p.N;
          const size_t rbase = ((size_t)a * p.N + (row_ok ? row : 0)) * p.K + (size_t)nt * BN + col_base;
          [[maybe_unused]] const size_t total = (size_t)p.G * p.N * p.K;
#pragma unroll
          for (int i = 0; i < EPI_COLS / 8; ++i) {
            const bool in = row_ok && nt * BN + col_base + i * 8 < p.K && AWQ_IN(rbase + i * 8, 8, total);
            d[i] = in ? *reinterpret_cast<const uint4*>(p.op + rbase + i * 8) : make_uint4(0u, 0u, 0u, 0u);
          }
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&tfull[buf], (ph >> buf) & 1u, p.timeout_ns, abort_flag, p.status)))
            return false;
          tc_fence_after();
          const uint32_t acc_addr = tmem_base + lane_base + (uint32_t)(buf * BN + col_base);
          float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
          for (int c = 0; c < EPI_COLS / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(acc_addr + (uint32_t)(c * 32), v);
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
            s0 = dot_bf16x8(f, d[4 * c], s0);
            s1 = dot_bf16x8(f + 8, d[4 * c + 1], s1);
            s0 = dot_bf16x8(f + 16, d[4 * c + 2], s0);
            s1 = dot_bf16x8(f + 24, d[4 * c + 3], s1);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[buf]);
          const float lane_sum = s0 + s1;
          if (p.row_acc != nullptr && row_ok && AWQ_IN((size_t)a * p.N + row, 1, (size_t)p.G * p.N))
            atomicAdd(&p.row_acc[(size_t)a * p.N + row], (double)lane_sum);
          item_sum += lane_sum;
        } else {
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&tfull[buf], (ph >> buf) & 1u, p.timeout_ns, abort_flag, p.status)))
            return false;
          tc_fence_after();
          const uint32_t acc_addr = tmem_base + lane_base + (uint32_t)(buf * BN + col_base);
          const float scale = nt < (mt >> 1) ? 2.0f : 1.0f;
          [[maybe_unused]] const size_t total = (size_t)p.K * p.K;
#pragma unroll 1
          for (int c = 0; c < EPI_COLS / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(acc_addr + (uint32_t)(c * 32), v);
            const int col0 = nt * BN + col_base + c * 32;
            if (col0 < p.K && row < p.K) {
              const size_t off = (size_t)row * p.K + col0;
              if (AWQ_IN(off, 32, total)) {
                uint4* dst = reinterpret_cast<uint4*>(p.H + off);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  dst[i] = make_uint4(pack_bf16x2(scale * __uint_as_float(v[8 * i]), scale * __uint_as_float(v[8 * i + 1])),
                                      pack_bf16x2(scale * __uint_as_float(v[8 * i + 2]), scale * __uint_as_float(v[8 * i + 3])),
                                      pack_bf16x2(scale * __uint_as_float(v[8 * i + 4]), scale * __uint_as_float(v[8 * i + 5])),
                                      pack_bf16x2(scale * __uint_as_float(v[8 * i + 6]), scale * __uint_as_float(v[8 * i + 7])));
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[buf]);
        }
        ph ^= 1u << buf;
        ++local;
      }
      if constexpr (LOSS) {
        if (last) {
          float ss = item_sum;
#pragma unroll
          for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
          [[maybe_unused]] const size_t n_part = (size_t)p.G * p.per_alpha * EPI_WARPS;
          if (lane == 0 && AWQ_IN((size_t)flat * EPI_WARPS + ew, 1, n_part))
            p.partials[(size_t)flat * EPI_WARPS + ew] = ss;
        }
      }
      return true;
    });
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- transpose
//
// Xt[j][t] = X[t][j] for t < n_tok and 0 for n_tok <= t < n_pad, in tiles of
// 64 tokens x 64 channels: 16-byte loads along the channels of X, 16-byte
// stores along the tokens of Xt, through a padded shared tile (66 halves a
// row, so that neither pass has bank conflicts).
constexpr int kTT = 64;

__global__ void __launch_bounds__(256) transpose_kernel(const uint16_t* __restrict__ X, int n, int K, int n_pad,
                                                        uint16_t* __restrict__ Xt) {
  __shared__ uint32_t tile[kTT * (kTT + 2) / 2];
  uint16_t* th = reinterpret_cast<uint16_t*>(tile);
  const int t0 = blockIdx.x * kTT, j0 = blockIdx.y * kTT;
  [[maybe_unused]] const size_t total_x = (size_t)n * K, total_t = (size_t)K * n_pad;
  for (int v = threadIdx.x; v < kTT * kTT / 8; v += blockDim.x) {
    const int r = v >> 3, c8 = (v & 7) * 8;
    const int t = t0 + r;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    const size_t off = (size_t)t * K + j0 + c8;
    if (t < n && AWQ_IN(off, 8, total_x)) val = *reinterpret_cast<const uint4*>(X + off);
    uint32_t* dst = tile + (r * (kTT + 2) + c8) / 2;
    dst[0] = val.x;
    dst[1] = val.y;
    dst[2] = val.z;
    dst[3] = val.w;
  }
  __syncthreads();
  for (int v = threadIdx.x; v < kTT * kTT / 8; v += blockDim.x) {
    const int jr = v & (kTT - 1), tc = (v >> 6) * 8;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = (uint32_t)th[(tc + 2 * i) * (kTT + 2) + jr] | ((uint32_t)th[(tc + 2 * i + 1) * (kTT + 2) + jr] << 16);
    const size_t off = (size_t)(j0 + jr) * n_pad + t0 + tc;
    if (AWQ_IN(off, 8, total_t)) *reinterpret_cast<uint4*>(Xt + off) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <bool LOSS>
cudaError_t launch_gram_kernel(const CUtensorMap& tmA, const CUtensorMap& tmB, const GramParams& p, int work,
                               cudaStream_t st) {
  cudaError_t e = ensure_dynamic_smem((const void*)gram_kernel<LOSS>, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  const int grid = work < sms ? work : sms;
  gram_kernel<LOSS><<<grid, NUM_THREADS, SMEM_BYTES, st>>>(tmA, tmB, p);
  return cudaGetLastError();
}

uint64_t timeout_of(const awq_config* cfg) {
  const uint32_t ms = cfg != nullptr && cfg->wait_timeout_ms ? cfg->wait_timeout_ms : 2000u;
  return (uint64_t)ms * 1000000ull;
}

}  // namespace

cudaError_t launch_gram_matrix(const uint16_t* X, int64_t n_tok, int64_t K, uint16_t* xt, uint16_t* H,
                               uint32_t* status, uint32_t wait_timeout_ms, cudaStream_t st) {
  const int64_t n_pad = gram_tokens_padded(n_tok);
  if (K / kTT > 65535) return cudaErrorInvalidValue;  // grid y
  transpose_kernel<<<dim3((unsigned)(n_pad / kTT), (unsigned)(K / kTT)), 256, 0, st>>>(X, (int)n_tok, (int)K,
                                                                                      (int)n_pad, xt);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap tmA, tmB;
  const cuuint64_t d[2] = {(cuuint64_t)n_pad, (cuuint64_t)K};
  const cuuint32_t ba[2] = {(cuuint32_t)BK, (cuuint32_t)BM};
  const cuuint32_t bb[2] = {(cuuint32_t)BK, (cuuint32_t)BN};
  if (!make_map(&tmA, xt, 2, d, ba) || !make_map(&tmB, xt, 2, d, bb)) return cudaErrorInvalidValue;
  GramParams p = {};
  p.K = (int)K;
  p.kb_tok = (int)(n_pad / BK);
  const int ct = (int)(K / BM);  // K is a multiple of 128
  const int m = ct / 2, b = ct % 2;
  p.items = (m + 1) * (m + b);
  awq_config c = {};
  c.wait_timeout_ms = wait_timeout_ms;
  p.timeout_ns = timeout_of(&c);
  p.status = status;
  p.H = H;
  return launch_gram_kernel<false>(tmA, tmB, p, p.items, st);
}

cudaError_t launch_gram_loss(const uint16_t* op, int64_t N, int64_t K, const awq_config& cfg, const uint16_t* H,
                             float* partials, uint32_t* status, cudaStream_t st, double* row_acc,
                             int withhold_first_fill) {
  CUtensorMap tmA, tmB;
  const cuuint64_t da[3] = {(cuuint64_t)K, (cuuint64_t)N, (cuuint64_t)cfg.n_grid};
  const cuuint32_t ba[3] = {(cuuint32_t)BK, (cuuint32_t)BM, 1u};
  const cuuint64_t dh[2] = {(cuuint64_t)K, (cuuint64_t)K};
  const cuuint32_t bh[2] = {(cuuint32_t)BK, (cuuint32_t)BN};
  if (!make_map(&tmA, op, 3, da, ba) || !make_map(&tmB, H, 2, dh, bh)) return cudaErrorInvalidValue;
  GramParams p = {};
  p.K = (int)K;
  p.N = (int)N;
  p.G = cfg.n_grid;
  p.nC = (int)((K + BN - 1) / BN);
  p.kbK = (int)(K / BK);
  p.nR = (int)((N + BM - 1) / BM);
  p.nP = (p.nC + 1) / 2;
  p.per_alpha = p.nR * p.nP;
  p.timeout_ns = timeout_of(&cfg);
  p.status = status;
  p.op = op;
  p.partials = partials;
  p.row_acc = row_acc;
  p.withhold_first_fill = withhold_first_fill;
  const int64_t items = (int64_t)p.G * p.per_alpha;
  return launch_gram_kernel<true>(tmA, tmB, p, items < (1 << 30) ? (int)items : (1 << 30), st);
}

#ifdef AWQ_CHECKED
cudaError_t take_oob_gram(unsigned long long* out) { return take_oob_record(out); }
#endif

}  // namespace awq
