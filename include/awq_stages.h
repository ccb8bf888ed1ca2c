/*
 * awq_stages.h - the kernels of step 2 of include/awq.h, one entry point
 * each. awq_search_layer runs awq_alpha_scales, then either awq_search_fused
 * or awq_fakequant followed by awq_search_gemm, then awq_loss_select, on its
 * workspace. These calls exist so that each kernel can be timed and checked
 * on its own; a user of the library needs only awq.h. Same conventions as
 * awq.h: device pointers, caller-owned buffers, 16-byte alignment,
 * asynchronous on `stream`, argument errors returned before any launch.
 */
#ifndef AWQ_B300_STAGES_H
#define AWQ_B300_STAGES_H

#include "awq.h"

#ifdef __cplusplus
extern "C" {
#endif

/* awq_search_layer (RESIDUAL form) runs the fake-quant inside the CTA-pair
   search kernel (awq_search_fused) when the search's products take fewer
   than this many flops, 2 * n_grid * n_tok * out * in. Larger searches run
   long enough to settle at the GPU's power limit, where the single-CTA
   products draw less energy per flop: they run awq_fakequant, then
   awq_search_gemm, whose products are the single-CTA kernel at that size. */
#define AWQ_SEARCH_FUSED_MAX_FLOPS 2e13

/* s[i][j] and inv_s[i][j] = 1/s[i][j] for every alpha_i (device fp32
   [n_grid][in]); the scale law of the search_scale listing and "AWQ >
   Summary", "The scaling formula". s is formed in fp64 (b^(i/n_grid) as the
   i-th power of b^(1/n_grid), times the fp64 reciprocal normaliser) and
   rounded to fp32 once; inv_s is the correctly rounded fp32 reciprocal of
   that value. */
AWQ_API awq_status awq_alpha_scales(const float* mean_abs, int64_t in, const awq_config* cfg, float* s,
                                    float* inv_s, awq_stream_t stream);

/* For every alpha_i: W_hat_i = Q(W * s_i) * inv_s_i (the scale, quantise and
   fold-back step of the search_scale listing; "AWQ > Salient Weight
   Preservation", scaling equation). RESIDUAL form writes bf16(W_hat_i - W)
   to op[i]; REFERENCE form writes bf16(W_hat_i) to op[i] and bf16(W) to
   op[n_grid]. op: device bf16 bits [n_slots][out][in]. */
AWQ_API awq_status awq_fakequant(const void* W, int32_t w_dtype, int64_t out, int64_t in, const float* s,
                                 const float* inv_s, const awq_config* cfg, uint16_t* op, awq_stream_t stream);

/* Tile grid of the search product: the n_tok x out output of one alpha is
   cut into m_tiles x n_tiles tiles of tile_m x tile_n. Host-only. */
AWQ_API awq_status awq_search_tiles(int64_t n_tok, int64_t out, const awq_config* cfg, int64_t* m_tiles,
                                    int64_t* n_tiles, int32_t* tile_m, int32_t* tile_n);

/* partials[i][mt][nt][q] = sum over the 32 tokens of lane quarter q of tile
   (mt, nt) and over the tile's outputs of (X op_i^T)^2 (RESIDUAL) or of
   (X op_i^T - X op_G^T)^2 (REFERENCE). X: device bf16 [n_tok][in]. op: as
   written by awq_fakequant. partials: device fp32 [n_grid][m_tiles][n_tiles][4].
   status: device uint32, set to AWQ_ERR_TIMEOUT if a wait ran out.
   tcgen05 tensor cores (bf16 in, fp32 accumulate in tensor memory), operands
   staged by TMA. The RESIDUAL form runs the products awq_search_layer runs
   for this size: CTA pairs (cta_group::2) below AWQ_SEARCH_FUSED_MAX_FLOPS,
   single CTAs from there on; the REFERENCE form runs on single CTAs. */
AWQ_API awq_status awq_search_gemm(const void* X, int64_t n_tok, int64_t in, const uint16_t* op, int64_t out,
                                   const awq_config* cfg, float* partials, uint32_t* status, awq_stream_t stream);

/* awq_fakequant followed by awq_search_gemm (RESIDUAL form only), in one
   kernel: besides the search roles, every CTA of the CTA-pair search kernel
   runs quantiser warps that write op (bit for bit what awq_fakequant writes)
   in the order the products consume it, one 256-row operand tile and
   512-channel strip at a time, and publish each tile in ready[i][nt]; the
   search waits (bounded) for a tile's counter before loading it, so the
   fake-quant overlaps the products instead of preceding them.
   W: device [out][in] (AWQ_BF16 or AWQ_FP32). s, inv_s: as written by
   awq_alpha_scales. op: device bf16 bits [n_grid][out][in] (scratch, fully
   written). partials, status: as awq_search_gemm. ready: device uint32
   scratch of n_grid * (n_tiles + 1) + 1 words (n_tiles from
   awq_search_tiles): per-tile and per-alpha counters and a progress word
   (the highest alpha started, plus one); zeroed by the call.
   Returns AWQ_ERR_UNSUPPORTED for the REFERENCE form. The quantiser warps of
   one CTA serve tiles consumed by others, so all CTAs of the launch must be
   resident together, as they are when the GPU runs nothing else (the grid is
   sized to the SM count); otherwise a wait runs out and *status reports
   AWQ_ERR_TIMEOUT. */
AWQ_API awq_status awq_search_fused(const void* W, int32_t w_dtype, int64_t out, int64_t in, const void* X,
                                    int64_t n_tok, const float* s, const float* inv_s, const awq_config* cfg,
                                    uint16_t* op, float* partials, uint32_t* ready, uint32_t* status,
                                    awq_stream_t stream);

/* Sizes of the GRAM form's buffers (elements): xt, the transposed copy of X
   (bf16 [in][n_pad], n_pad = n_tok rounded up to 64); H (bf16 [in][in]);
   partials per alpha (fp32). Host-only. */
AWQ_API awq_status awq_gram_sizes(int64_t n_tok, int64_t out, int64_t in, int64_t* xt_elems, int64_t* h_elems,
                                  int64_t* partials_per_alpha);

/* H[c][j] = bf16(f * sum_t X[t][c] X[t][j]) for the 256-channel blocks
   jb(j) <= jb(c) (f = 2 below the block diagonal, 1 on it; the blocks above
   it are not written): the Gram matrix of the GRAM loss form, fp32
   accumulation on tcgen05 tensor cores. X: device bf16 [n_tok][in]. xt:
   device scratch of awq_gram_sizes' xt_elems bf16 (overwritten with X^T,
   zero past n_tok). H: device bf16 [in][in]. status: as awq_search_gemm. */
AWQ_API awq_status awq_gram_matrix(const void* X, int64_t n_tok, int64_t in, uint16_t* xt, uint16_t* H,
                                   const awq_config* cfg, uint32_t* status, awq_stream_t stream);

/* The GRAM form's per-alpha sums: for every alpha_i, partial sums of
   sum_r sum_c op_i[r][c] sum_{j: jb(j) <= jb(c)} H[c][j] op_i[r][j]
   = sum_r op_i[r] (X^T X) op_i[r]^T (op_i = bf16(W_hat_i - W) from
   awq_fakequant, RESIDUAL form; H from awq_gram_matrix), as
   partials[i][awq_gram_sizes' partials_per_alpha] (fp32). The alphas'
   products run on tcgen05 tensor cores, 128 x 256 tiles over each tile's
   prefix of channel blocks, their epilogue adding product x op_i. */
AWQ_API awq_status awq_gram_loss(const uint16_t* op, int64_t out, int64_t in, const uint16_t* H,
                                 const awq_config* cfg, float* partials, uint32_t* status, awq_stream_t stream);

/* losses[i] = (sum of partials[i]) / (n_tok * out), partials as written by
   awq_search_gemm (or, with cfg->loss_form GRAM, by awq_gram_loss): fp32
   sums per thread over a fixed stride, fp64 across threads in a fixed tree (deterministic);
   best_idx = first i with the smallest fp32 loss (the strict "<" of the
   search_scale listing); s_best = s[best_idx]. A non-finite loss sets
   *status to AWQ_ERR_NONFINITE. */
AWQ_API awq_status awq_loss_select(const float* partials, int64_t n_tok, int64_t out, int64_t in, const float* s,
                                   const awq_config* cfg, float* losses, int32_t* best_idx, float* s_best,
                                   uint32_t* status, awq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* AWQ_B300_STAGES_H */
