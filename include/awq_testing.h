/*
 * awq_testing.h - test aids of the library. None of these calls is part of
 * the method or needed to use it: they let the test suite look inside the
 * kernels (raw products), make a device-side wait run out on purpose (the
 * bounded waits end with a status, the GPU stays usable), and read the
 * record of the bounds-checked build. Conventions as in awq.h.
 */
#ifndef AWQ_B300_TESTING_H
#define AWQ_B300_TESTING_H

#include "awq.h"

#ifdef __cplusplus
extern "C" {
#endif

/* awq_search_gemm (include/awq_stages.h) in RESIDUAL form with a chosen
   kernel: single_cta 0 = the CTA-pair kernel awq_search_gemm uses
   (cta_group::2, two CTAs share each 256x256 tile, each loading its half of
   the operand tile); 1 = the single-CTA kernel. If `dump` is not NULL the
   kernel also stores the raw fp32 products D[i][t][r] = (X op_i^T)[t][r]
   there (device fp32 [n_grid][n_tok][out]), so the tensor-core data path can
   be checked element by element against a plain matrix product on small
   shapes; those stores cost n_grid * n_tok * out * 4 bytes of traffic. */
AWQ_API awq_status awq_search_gemm_dump(const void* X, int64_t n_tok, int64_t in, const uint16_t* op, int64_t out,
                                        const awq_config* cfg, float* partials, uint32_t* status, float* dump,
                                        int32_t single_cta, awq_stream_t stream);

/* The bounded waits of the GRAM form's products: awq_gram_loss with the
   first ring fill of every CTA left out, so the MMA issuer's wait on that
   stage can never complete. As for awq_search_gemm_withhold_fill: each wait
   gives up after cfg->wait_timeout_ms, the kernel writes AWQ_ERR_TIMEOUT to
   *status, stops all its roles, lets what it issued finish, frees its tensor
   memory and returns. partials are not meaningful. */
AWQ_API awq_status awq_gram_loss_withhold_fill(const uint16_t* op, int64_t out, int64_t in, const uint16_t* H,
                                               const awq_config* cfg, float* partials, uint32_t* status,
                                               awq_stream_t stream);

/* The bounded waits of the single-CTA search kernel: awq_search_gemm with
   the first operand fill of every CTA left out, so the MMA issuer's wait on
   that pipeline stage can never complete. Each wait gives up after
   cfg->wait_timeout_ms; the kernel then writes AWQ_ERR_TIMEOUT to *status,
   stops all its roles, lets the copies and MMAs it did issue finish, frees
   its tensor memory and returns, leaving the device usable. partials are not
   meaningful. */
AWQ_API awq_status awq_search_gemm_withhold_fill(const void* X, int64_t n_tok, int64_t in, const uint16_t* op,
                                                 int64_t out, const awq_config* cfg, float* partials,
                                                 uint32_t* status, awq_stream_t stream);

/* The cross-CTA waits of awq_search_fused: the quantiser warps leave out
   their first unit (alpha 0, operand tile 0, channel strip 0), so that
   tile's ready counter never completes and the TMA producers that need it
   wait in vain. Each wait gives up after cfg->wait_timeout_ms; the kernel
   then writes AWQ_ERR_TIMEOUT to *status, stops all its roles, lets what it
   issued finish, frees its tensor memory and returns. Same arguments as
   awq_search_fused; partials and op are not meaningful. */
AWQ_API awq_status awq_search_fused_withhold_unit(const void* W, int32_t w_dtype, int64_t out, int64_t in,
                                                  const void* X, int64_t n_tok, const float* s, const float* inv_s,
                                                  const awq_config* cfg, uint16_t* op, float* partials,
                                                  uint32_t* ready, uint32_t* status, awq_stream_t stream);

/* The library can be built with every global-memory access of its bandwidth
   kernels, quantiser warps, search epilogue and decode product preceded by a
   bounds check against the buffer's extent as the call's shapes define it
   (python -m post_bit_weight_awq_b300.build --checked, which writes
   libawq_checked.so next to libawq.so). A failed check is counted and its
   access skipped, so an indexing error shows up as a count instead of a
   memory fault. awq_bounds_report returns the number of failed checks since
   the previous report and, for the first recorded one, the source unit
   (1 awq_kernels.cu, 2 awq_search_gemm.cu, 3 awq_w4a16.cu, 4 awq_gram.cu;
   0 if none), line
   and element offset, then clears the records; it synchronises the device.
   awq_bounds_selftest launches one check that fails by construction (the
   element one past `buf[0..n)`; nothing is written). Both return
   AWQ_ERR_UNSUPPORTED from the release library. */
AWQ_API awq_status awq_bounds_report(uint64_t* failures, int32_t* unit, uint64_t* line, uint64_t* offset);
AWQ_API awq_status awq_bounds_selftest(float* buf, int32_t n, awq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* AWQ_B300_TESTING_H */
