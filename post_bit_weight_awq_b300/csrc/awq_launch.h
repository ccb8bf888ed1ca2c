// Internal host-side launchers shared by the C ABI (awq_api.cu) and the
// kernel translation units. Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "awq.h"

namespace awq {

constexpr int kBlockCols = 128;  // input channels of one 8-lane block of the quantiser kernels; `in` is a multiple
constexpr int kMaxGrid = 64;     // largest alpha grid
// Statistics: a block reads a strip of 256 channels over a chunk of tokens;
// the chunk length depends on the shape only (results do not depend on the
// GPU) and is chosen so that about kStatsTargetBlocks blocks cover X: one
// wave of 4 resident blocks on each SM of a 148-SM B300.
constexpr int kStatsTargetBlocks = 592;
constexpr int kStatsRowQuantum = 32;  // chunk lengths are multiples of 8 row phases x 4 rows per batch

// Search-product tiling (one CTA per SM, persistent).
constexpr int kTileM = 128;  // tokens per tile (tensor-memory lanes)
constexpr int kTileN = 256;  // output rows per tile (tensor-memory columns)
constexpr int kTileK = 64;   // input channels per pipeline stage (128 B of bf16)

// SM count of the current device, queried once per device.
cudaError_t sm_count(int* sms);
// Allow `bytes` of dynamic shared memory for kernel `func` on the current
// device (the attribute is set once per kernel, device and size increase).
cudaError_t ensure_dynamic_smem(const void* func, int bytes);
// TMA map of a bf16 tensor of rank 2 or 3 (dims innermost first, densely
// packed), 128-byte swizzle, zero fill outside the extents. False if the
// driver entry point is missing or the map cannot be encoded.
bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint32_t* box);

inline int stats_strips(int64_t in) { return (int)((in + 255) / 256); }
// Tokens per statistics chunk: the token range split into
// kStatsTargetBlocks / strips chunks (at least one), each rounded up to a
// multiple of kStatsRowQuantum, so that strips x chunks stays within
// kStatsTargetBlocks whenever there are fewer strips than that.
inline int64_t stats_chunk_rows(int64_t n_tok, int64_t in) {
  const int64_t strips = stats_strips(in);
  const int64_t target = strips < kStatsTargetBlocks ? kStatsTargetBlocks / strips : 1;
  const int64_t per = (n_tok + target - 1) / target;
  const int64_t q = (per + kStatsRowQuantum - 1) / kStatsRowQuantum * kStatsRowQuantum;
  return q < kStatsRowQuantum ? kStatsRowQuantum : q;
}
// Chunks of the token range: at most max(1, kStatsTargetBlocks / strips).
inline int stats_chunks(int64_t n_tok, int64_t in) {
  const int64_t r = stats_chunk_rows(n_tok, in);
  return (int)((n_tok + r - 1) / r);
}

// partials: fp32 [stats_chunks(n, K)][K]; tickets: uint32 [stats_strips(K)] (zeroed by the launch).
cudaError_t launch_stats(const uint16_t* X, int64_t n, int64_t K, float* partials, uint32_t* tickets,
                         float* mean_abs, cudaStream_t st);
cudaError_t launch_alpha_scales(const float* mean_abs, int64_t K, const awq_config& cfg, float* s,
                                float* inv_s, cudaStream_t st);
cudaError_t launch_fakequant(const void* W, int w_dtype, int64_t N, int64_t K, const float* s,
                             const float* inv_s, const awq_config& cfg, uint16_t* op, cudaStream_t st);
cudaError_t launch_pack(const void* W, int w_dtype, int64_t N, int64_t K, const float* s,
                        const awq_config& cfg, int32_t* qweight, uint16_t* scales, uint16_t* zeros,
                        cudaStream_t st);
// row_losses[i][r] = row_acc[i][r] / (n_tok * N) as fp32.
cudaError_t launch_row_losses(const double* row_acc, int G, int64_t N, int64_t n_tok, float* row_losses,
                              cudaStream_t st);

cudaError_t launch_loss_select(const float* partials, int G, int64_t per_alpha, int64_t n_tok, int64_t N,
                               const float* s, int64_t K, float* losses, int32_t* best_idx, float* s_best,
                               uint32_t* status, cudaStream_t st);

// Returns cudaErrorInvalidValue (without launching) if a tensor map cannot
// be encoded.
cudaError_t launch_search_gemm(const uint16_t* X, int64_t n_tok, int64_t K, const uint16_t* op, int64_t N,
                               const awq_config& cfg, float* partials, uint32_t* status, cudaStream_t st,
                               float* dump = nullptr, int withhold_first_fill = 0, int single_cta = 0,
                               double* row_acc = nullptr);
// single_cta: 0 = the default kernel (CTA pairs, cta_group::2, for the
// RESIDUAL form); 1 = the single-CTA kernel (always used for the REFERENCE
// form and the withheld-fill test aid).
// row_acc: if not null, fp64 [n_grid][N] to which each output row's sum of
// squared errors over the tokens is added (the caller zeroes it).

// Words of the fused search's synchronisation scratch: a counter per operand
// tile and per alpha, and one progress word.
inline size_t fused_ready_words(int64_t G, int64_t n_tiles) { return (size_t)(G * (n_tiles + 1) + 1); }

// RESIDUAL form with the fake-quant fused in: quantiser warps in every CTA of
// the CTA-pair search kernel write op (as launch_fakequant does) while the
// search consumes it. ready: uint32 [fused_ready_words(n_grid, ceil(N/256))],
// zeroed by the call.
cudaError_t launch_search_fused(const void* W, int w_dtype, const uint16_t* X, int64_t n_tok, int64_t K,
                                const float* s, const float* inv_s, int64_t N, const awq_config& cfg, uint16_t* op,
                                float* partials, uint32_t* ready, uint32_t* status, cudaStream_t st,
                                float* dump = nullptr, int skip_unit = -1, double* row_acc = nullptr);

// y[m][r] = sum_k x[m][k] * (q[r][k] - z[r][g]) * scale[r][g] for m < M <= 8,
// g = k / group (group 32, 64 or 128), x bf16 [M][K] (staged as fp32 in
// shared memory: M * K * 4 bytes).
cudaError_t launch_w4a16_gemv(const uint16_t* x, int64_t M, int64_t K, const int32_t* qweight, const uint16_t* scales,
                              const uint16_t* zeros, int64_t N, int group, float* y, cudaStream_t st);

#ifdef AWQ_CHECKED
// Checked builds: each kernel translation unit's record of failed bounds
// checks (count, first source line, first offset), read and zeroed.
cudaError_t take_oob_kernels(unsigned long long* out);
cudaError_t take_oob_search(unsigned long long* out);
cudaError_t take_oob_w4a16(unsigned long long* out);
cudaError_t take_oob_gram(unsigned long long* out);
cudaError_t launch_bounds_selftest(float* buf, int n, cudaStream_t st);
#endif

// Gram form of the search loss (awq_gram.cu). kGramRowGroup: 128-row blocks
// whose items for one column-block pair run on neighbouring CTAs.
#ifndef AWQ_GRAM_ROW_GROUP
#define AWQ_GRAM_ROW_GROUP 16
#endif
constexpr int kGramRowGroup = AWQ_GRAM_ROW_GROUP;
constexpr int kGramEpilogueWarps = 8;
inline int64_t gram_tokens_padded(int64_t n_tok) { return (n_tok + 63) / 64 * 64; }
// Column-block pairs (blocks cb and nC-1-cb of 256 channels) of in channels.
inline int64_t gram_pairs(int64_t K) { return ((K + 255) / 256 + 1) / 2; }
// fp32 partial sums of one alpha: [row blocks x pairs][epilogue warps].
inline int64_t gram_partials_per_alpha(int64_t N, int64_t K) {
  return (N + kTileM - 1) / kTileM * gram_pairs(K) * kGramEpilogueWarps;
}
// H (bf16 [K][K], blocks on and below the 256-channel block diagonal) of X
// (bf16 [n_tok][K], K a multiple of 128), through the transposed copy xt
// (bf16 [K][gram_tokens_padded(n_tok)], overwritten).
cudaError_t launch_gram_matrix(const uint16_t* X, int64_t n_tok, int64_t K, uint16_t* xt, uint16_t* H,
                               uint32_t* status, uint32_t wait_timeout_ms, cudaStream_t st);
// partials[a][...] of sum_r D_a[r] C D_a[r]^T, D_a = op slot a (bf16 [n_grid][N][K]).
// row_acc: if not null, fp64 [n_grid][N] to which each row's sum is added.
// withhold_first_fill: test aid, each CTA's first ring stage is never filled.
cudaError_t launch_gram_loss(const uint16_t* op, int64_t N, int64_t K, const awq_config& cfg, const uint16_t* H,
                             float* partials, uint32_t* status, cudaStream_t st, double* row_acc = nullptr,
                             int withhold_first_fill = 0);

// W_hat[r][k] = bf16((q[r][k] - z[r][g]) * scale[r][g]) for the whole packed
// layer (bf16 [N][K]), the operand of the prefill product.
cudaError_t launch_w4_expand(const int32_t* qweight, const uint16_t* scales, const uint16_t* zeros, int64_t N,
                             int64_t K, int group, uint16_t* w_hat, cudaStream_t st);

}  // namespace awq
