/*
 * awq.h - C ABI of the B300 (sm_103a) AWQ per-layer scale search and INT4 pack.
 *
 * What the library computes, for one linear layer with weights W[out, in] and
 * calibration activations X[n_tok, in]:
 *
 *   1. sx[j]   = mean_t |X[t, j]|                               (awq_act_stats)
 *   2. for alpha_i = i / n_grid, i = 0 .. n_grid-1:
 *        s_i[j]  = max(sx[j], sx_clamp_min) ^ alpha_i, optionally divided by
 *                  sqrt(max_j s_i * min_j s_i)
 *        W_hat_i = Q(W * diag(s_i)) * diag(1 / s_i)
 *        L_i     = mean over (t, r) of (X W_hat_i^T - X W^T)[t, r]^2
 *      best = first i with the smallest L_i                     (awq_search_layer)
 *   3. codes of W * diag(s_best) packed 8 per int32 (32/w_bit for 2 or 8
 *      bits), fp16 group scales and fp16 zero points           (awq_quantize_pack)
 *   4. the packed layer applied to activations: a few tokens   (awq_w4a16_gemv)
 *      or any number of tokens                                  (awq_w4a16_gemm)
 * Steps 1-3 for a sequence of layers held in host memory, with the copies
 * overlapping the work: awq_quantize_layers. Several linears that read one X
 * and must share one s: awq_search_block.
 *
 * Q is group-wise asymmetric min/max quantisation along `in` (groups of
 * `group` weights): delta = max((vmax - vmin) / (2^w_bit - 1), delta_floor),
 * z = rne(-vmin / delta), q = clamp(rne(v / delta) + z, 0, 2^w_bit - 1),
 * dequantised value (q - z) * delta. Codes are decided in fp32 with correctly
 * rounded operations in exactly that order; rne is round-half-to-even. With
 * zero_point = 0 Q is the symmetric round-to-nearest of "Why does naive
 * 4-bit quantization wreck LLM accuracy?" on the first page:
 * delta = max(max|v| / 2^(w_bit-1), delta_floor), z = 2^(w_bit-1) fixed,
 * same q and dequantisation (the top code clamps at 2^(w_bit-1) - 1 steps).
 *
 * Sources (web pages on AWQ, by title and section):
 *   - "AWQ: How Activation-Aware Quantization Saves 4-bit LLMs":
 *     "How does AWQ decide which weights to protect?" (mean |x| per input
 *     channel), "How does AWQ protect channels without mixed precision?" (the
 *     alpha grid search over s = sx^alpha against the output MSE of the
 *     unquantised layer), and the deployment quant_config (4 bits, groups of
 *     128, zero point on).
 *   - "AWQ > Salient Weight Preservation": the step-size equation (range over
 *     2^b - 1 levels) and the scaling equation (w*s times x/s leaves y alone).
 *   - "AWQ > Summary": "The scaling formula" (alpha) and "Salient weight
 *     identification" (mean absolute activation).
 *   - "What is AWQ Quantization? Definition & 4-Bit Weight Compression in
 *     Enterprise AI", step "INT4 Weight Packing & Export" (INT32 containers).
 *   - "AWQ (Activation-Aware Weight Quantization) - AI Glossary", "Example:
 *     Where 4-bit memory saving comes from" (one 16-bit scale per 128 weights).
 *   The normalisation by sqrt(max * min) is not on the pages; it is part of
 *   this library's specification and, in exact arithmetic, does not change
 *   W_hat_i.
 *
 * Conventions for every call below:
 *   - Pointers named X, W, s, mean_abs, losses, ... are DEVICE pointers unless
 *     the comment says host. The caller owns every buffer; the library
 *     allocates no device memory. Scratch memory comes from the caller through
 *     `ws` / `ws_bytes`, sized with the *_workspace_size queries.
 *   - Matrices are dense row-major: X[n_tok][in], W[out][in]; `in` is the
 *     contiguous dimension. Device pointers must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream). Argument errors are detected on the host and returned
 *     before anything is launched. Launch failures return AWQ_ERR_CUDA.
 *     Conditions found on the device (a bounded wait that ran out, a
 *     non-finite loss) are written to a device status word; read it with
 *     awq_get_device_status, which synchronises the stream.
 *   - Shapes: group 32, 64 or 128 ("AWQ: How Activation-Aware Quantization
 *     Saves 4-bit LLMs", deployment notes: finer groups, more scales), in a
 *     multiple of 128 whatever the group (the kernels hold 128-channel
 *     blocks in 8 lanes), w_bit 2..8 for the search, 2, 4 or 8 for
 *     awq_quantize_pack and 4 for the products over the packed layer
 *     (awq_w4a16_gemv, awq_w4a16_gemm), zero_point 0 or 1,
 *     1 <= n_grid <= 64. Other group sizes and widths return
 *     AWQ_ERR_UNSUPPORTED. n_tok and out are arbitrary (>= 1); the loss
 *     divides by the true n_tok * out.
 *   - The codes quantise W * diag(s): the caller folds 1/s into whatever
 *     produces X (for a transformer, the preceding LayerNorm/RMSNorm weight,
 *     as "AWQ > Salient Weight Preservation" describes). s_best is returned
 *     for that purpose.
 */
#ifndef AWQ_B300_H
#define AWQ_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define AWQ_API __attribute__((visibility("default")))
#else
#define AWQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t, declared here so the header needs no CUDA
   include. */
typedef struct CUstream_st* awq_stream_t;

typedef enum {
  AWQ_OK = 0,
  AWQ_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad config */
  AWQ_ERR_UNSUPPORTED = 2, /* valid but not built: group not 32/64/128, w_bit outside 2..8 (2/4/8 to pack) ... */
  AWQ_ERR_MISALIGNED = 3,  /* a device pointer is not 16-byte aligned */
  AWQ_ERR_WORKSPACE = 4,   /* ws_bytes below the size the query returns */
  AWQ_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
  AWQ_ERR_TIMEOUT = 6,     /* device: a bounded wait ran out; results invalid */
  AWQ_ERR_NONFINITE = 7    /* device: a loss was NaN or Inf */
} awq_status;

typedef enum { AWQ_BF16 = 0, AWQ_FP32 = 1 } awq_dtype;

/* How the search scores each alpha. All give the same number in exact
   arithmetic, since X W_hat^T - X W^T = X (W_hat - W)^T and
   sum_t sum_r (X D^T)[t][r]^2 = sum_r D[r] (X^T X) D[r]^T.
   RESIDUAL:  one bf16 product per alpha, X (W_hat - W)^T, squared and summed
              in the GEMM epilogue: 2 n_tok out in flops per alpha (default).
   REFERENCE: the output X W^T of the unquantised weight is computed once per
              output tile, kept resident in tensor memory, and subtracted from
              X W_hat^T in the epilogue, as the search_scale listing of the
              first page writes it.
   GRAM:      C = X^T X is formed once per search (fp32 accumulation, kept as
              bf16, only the 256-channel blocks on and below the diagonal),
              then each alpha costs out in^2 flops: P = D C over each output
              tile's prefix of channel blocks, and the epilogue adds
              P[r][c] * D[r][c]. Fewer flops than RESIDUAL when in < 2 n_tok.
              The losses differ from RESIDUAL's by the bf16 rounding of C
              (about 2^-9 / sqrt(in) relative when C's diagonal dominates).
              in <= 65535 * 64 (else AWQ_ERR_UNSUPPORTED); the workspace
              holds C, in * in bf16.
   AUTO:      GRAM when its tensor-core flops (C plus the alphas' products)
              are below 0.7 of RESIDUAL's and in <= 65535 * 64, else
              RESIDUAL (default). The choice
              depends on the shape and n_grid only; awq_search_form reports it.
              The per-kernel calls of awq_stages.h take AUTO as RESIDUAL. */
typedef enum {
  AWQ_LOSS_RESIDUAL = 0,
  AWQ_LOSS_REFERENCE = 1,
  AWQ_LOSS_GRAM = 2,
  AWQ_LOSS_AUTO = 3
} awq_loss_form;

typedef struct {
  int32_t w_bit;            /* 4: bits per code (2..8 in the search; 2, 4 or 8 packed; 4 in the products) */
  int32_t group;            /* 128: weights per scale/zero along `in` (32, 64 or 128) */
  int32_t n_grid;           /* 20: alpha_i = i / n_grid, i < n_grid */
  int32_t zero_point;       /* 1: asymmetric with zero point; 0: symmetric, delta = max|v| / 2^(w_bit-1),
                               codes stored with the fixed zero point 2^(w_bit-1) */
  int32_t normalize;        /* 1: divide s by sqrt(max(s) * min(s)) */
  float sx_clamp_min;       /* 1e-4: sx is clamped from below before the power */
  float delta_floor;        /* 1e-5: lower bound of a group's step */
  int32_t loss_form;        /* awq_loss_form (AUTO) */
  uint32_t wait_timeout_ms; /* bound of each device-side wait; 0 = 2000 ms */
} awq_config;

/* Fill `cfg` with the defaults above. */
AWQ_API void awq_config_default(awq_config* cfg);

/* Static, NUL-terminated description of a status; never NULL. */
AWQ_API const char* awq_status_string(int status);

/* ---------------------------------------------------------------- step 1 */

/* Device bytes of scratch that awq_act_stats needs for (n_tok, in). Host-only.
   Returns AWQ_ERR_INVALID_ARG for non-positive sizes or a NULL `bytes`. */
AWQ_API awq_status awq_act_stats_workspace_size(int64_t n_tok, int64_t in, size_t* bytes);

/* mean_abs[j] = (1/n_tok) sum_t |X[t, j]|  (fp32 out; fp32 partial sums over
   chunks of tokens whose length depends only on n_tok and in, a compensated
   fp32 sum across chunks, fixed order: deterministic). One kernel, preceded
   by a small memset of the scratch's ticket counters on `stream`.
   X: device bf16 [n_tok][in] (x_dtype must be AWQ_BF16). in % 8 == 0.
   mean_abs: device fp32 [in]. ws: device scratch of at least the queried
   size. Source: "AWQ: How Activation-Aware Quantization Saves 4-bit LLMs",
   "How does AWQ decide which weights to protect?"; "AWQ > Summary",
   "Salient weight identification". */
AWQ_API awq_status awq_act_stats(const void* X, int32_t x_dtype, int64_t n_tok, int64_t in,
                         float* mean_abs, void* ws, size_t ws_bytes, awq_stream_t stream);

/* Largest number of fp32 partial sums (chunks * in, with
   max(1, 592 / ceil(in / 256)) chunks of tokens at most) that
   awq_act_stats_noalloc accepts: its fixed scratch holds 4 MiB of partial
   sums plus 16 KiB of counters. Every n_tok is accepted for in up to 2^20
   channels. */
#define AWQ_NOALLOC_STATS_MAX_FLOATS (1u << 20)

/* awq_act_stats for callers that cannot allocate device memory or pass a
   scratch buffer (for example a plugin inside an engine that owns all device
   memory and gives the plugin only its inputs and outputs, or a path where a
   cudaMalloc, which may synchronise the device, is not allowed). The pages
   have no counterpart: this is an interface variant of step 1, not part of
   the method. Same arguments and result as awq_act_stats without ws/ws_bytes.
   The partial sums live in a library-owned device array (4 MiB + 16 KiB)
   that every GPU loading the library keeps until exit; each call clears the
   array's counters with a memset on `stream` before its kernel. Its address
   is looked up on the first call made in each context of a device (with that
   device current), so after a cudaDeviceReset the next call looks it up
   again; make the first call on a device before any stream capture. All
   calls share the array, so calls that overlap on the GPU race: serialise
   them. Calls allocate nothing. Returns AWQ_ERR_WORKSPACE if the partial
   sums exceed AWQ_NOALLOC_STATS_MAX_FLOATS. */
AWQ_API awq_status awq_act_stats_noalloc(const void* X, int32_t x_dtype, int64_t n_tok, int64_t in,
                                         float* mean_abs, awq_stream_t stream);

/* ---------------------------------------------------------------- step 2 */

/* Device bytes of scratch that awq_search_layer needs. Host-only. It holds a
   status word, s and 1/s for every alpha ([n_grid][in] fp32 each), the bf16
   search operand for every alpha ([n_grid (+1 in REFERENCE form)][out][in]),
   the per-tile partial sums and the operand-tile ready counters; in GRAM
   form also X^T X as bf16 [in][in] (X^T itself shares the operand's space). */
AWQ_API awq_status awq_workspace_size(int64_t n_tok, int64_t out, int64_t in, const awq_config* cfg,
                              size_t* bytes);

/* The loss form awq_search_layer runs for this shape and configuration:
   cfg->loss_form itself, or for AWQ_LOSS_AUTO the form it resolves to
   (AWQ_LOSS_GRAM or AWQ_LOSS_RESIDUAL). Host-only. */
AWQ_API awq_status awq_search_form(int64_t n_tok, int64_t out, int64_t in, const awq_config* cfg, int32_t* form);

/* The alpha grid search of "AWQ: How Activation-Aware Quantization Saves
   4-bit LLMs", "How does AWQ protect channels without mixed precision?"
   (search_scale listing), with the quantiser above.
   W: device [out][in], w_dtype AWQ_BF16 or AWQ_FP32. X: device bf16
   [n_tok][in] (x_dtype AWQ_BF16). mean_abs: device fp32 [in] (from step 1).
   losses: device fp32 [n_grid], the mean squared output error per alpha.
   best_idx: device int32 [1], first index of the smallest loss.
   s_best: device fp32 [in], s of that alpha (fold 1/s_best into X's producer).
   row_losses: NULL, or device fp32 [n_grid][out]: each output row's share of
   the loss, sum over tokens of the squared error of that row divided by
   n_tok * out (so a row of row_losses sums to the loss up to rounding); the
   search epilogue adds them up in fp64 as it goes, at some extra cost.
   ws/ws_bytes: scratch, at least awq_workspace_size(); its first 4 bytes are
   the device status word read by awq_get_device_status.
   The products run on bf16 tensor cores with fp32 accumulation; the step-2
   output matrix never leaves the chip. The kernels it runs, each also
   callable alone, are declared in awq_stages.h. */
AWQ_API awq_status awq_search_layer(const void* W, int32_t w_dtype, int64_t out, int64_t in,
                            const void* X, int32_t x_dtype, int64_t n_tok, const float* mean_abs,
                            const awq_config* cfg, float* losses, int32_t* best_idx,
                            float* s_best, float* row_losses, void* ws, size_t ws_bytes,
                            awq_stream_t stream);

/* Several linears that read the same input X (the q/k/v projections behind
   one RMSNorm, or gate/up behind another) must share one s, because 1/s is
   folded into that one producer of X ("AWQ > Salient Weight Preservation":
   the inverse scale is absorbed into the preceding LayerNorm/RMSNorm). The
   block search scores each alpha by the output MSE of all the linears
   together, i.e. the search of the layer whose weight is their rows one
   after another: L_i = sum_j sum (X W_hat_ij^T - X W_j^T)^2 / (n_tok *
   sum_j out_j). At most AWQ_BLOCK_MAX_LINEARS linears. */
#define AWQ_BLOCK_MAX_LINEARS 16

/* Device bytes of scratch awq_search_block needs: awq_workspace_size for
   sum_j outs[j] rows plus room for those rows of W. Host-only; outs is a
   host array of `count` output sizes. */
AWQ_API awq_status awq_search_block_workspace_size(int64_t n_tok, const int64_t* outs, int32_t count, int64_t in,
                                                   int32_t w_dtype, const awq_config* cfg, size_t* bytes);

/* awq_search_layer over a block of linears sharing X. W_list: HOST array of
   `count` device pointers, W_list[j] of [outs[j]][in] (same dtype, 16-byte
   aligned); outs: HOST array. The rows are copied one after another into the
   workspace (device-to-device copies on `stream`), then searched as one
   layer. Outputs as awq_search_layer; pack each linear afterwards with
   awq_quantize_pack and the same s_best. */
AWQ_API awq_status awq_search_block(const void* const* W_list, int32_t w_dtype, const int64_t* outs, int32_t count,
                                    int64_t in, const void* X, int32_t x_dtype, int64_t n_tok,
                                    const float* mean_abs, const awq_config* cfg, float* losses, int32_t* best_idx,
                                    float* s_best, void* ws, size_t ws_bytes, awq_stream_t stream);

/* ---------------------------------------------------------------- step 3 */

/* Final INT4 codes of W * diag(s) with the quantiser above, bit-exact with
   respect to fp32 arithmetic ("What is AWQ Quantization? ...", "INT4 Weight
   Packing & Export"; "AWQ (Activation-Aware Weight Quantization) - AI
   Glossary", memory example).
   W: device [out][in] (AWQ_BF16 or AWQ_FP32). s: device fp32 [in].
   qweight: device int32 [out][in/8]; the code of column 8j+k sits in bits
   [4k, 4k+4) of word j. scales_f16 / zeros_f16: device fp16 bit patterns
   [out][in/group] holding fp16(delta) and fp16(z), round-to-nearest-even.
   cfg->w_bit 4 is the pages' format (4-bit codes in INT32 containers); 2 and
   8 pack the same way, 16 or 4 codes to a word: qweight is then int32
   [out][in * w_bit / 32], column (32/w_bit) j + k in bits
   [w_bit k, w_bit k + w_bit) of word j. Other widths (3, 5, 6, 7 do not fill
   a 32-bit word evenly) return AWQ_ERR_UNSUPPORTED. Needs no scratch. */
AWQ_API awq_status awq_quantize_pack(const void* W, int32_t w_dtype, int64_t out, int64_t in,
                             const float* s, const awq_config* cfg, int32_t* qweight,
                             uint16_t* scales_f16, uint16_t* zeros_f16, awq_stream_t stream);

/* The packed layer applied to any number of tokens (the prefill case; for
   up to AWQ_W4A16_MAX_TOKENS tokens awq_w4a16_gemv reads the codes
   directly). The layer is expanded once into the workspace as
   W_hat[r][k] = bf16((q - z[r][g]) * scale[r][g]) (the fp32 product is
   exact while |q - z| < 2^13, so bf16 rounding is its only approximation:
   at most 2^-8 relative per weight), then y = x W_hat^T runs on the tensor
   cores with fp32 accumulation (the search's CTA-pair product with one
   operand). x: device bf16 [n_tok][in]; y: device fp32 [n_tok][out],
   16-byte aligned; ws: awq_w4a16_gemm_workspace_size() bytes, its first 4
   bytes a status word (awq_get_device_status). cfg->w_bit must be 4. */
AWQ_API awq_status awq_w4a16_gemm_workspace_size(int64_t n_tok, int64_t in, int64_t out, const awq_config* cfg,
                                                 size_t* bytes);
AWQ_API awq_status awq_w4a16_gemm(const void* x, int32_t x_dtype, int64_t n_tok, int64_t in,
                                  const int32_t* qweight, const uint16_t* scales_f16, const uint16_t* zeros_f16,
                                  int64_t out, const awq_config* cfg, float* y, void* ws, size_t ws_bytes,
                                  awq_stream_t stream);

/* ---------------------------------------------------------------- layers from host memory */

/* One layer of awq_quantize_layers. Pointers may be host or device memory
   (unified addressing); host buffers should be pinned (cudaHostAlloc or
   cudaHostRegister) for the copies to overlap the computation. */
typedef struct {
  const void* W;        /* [out][in], of the call's w_dtype */
  const void* X;        /* bf16 [n_tok][in]: the layer's calibration activations */
  int64_t n_tok, out, in;
  int32_t* qweight;     /* out: [out][in * w_bit / 32], as awq_quantize_pack */
  uint16_t* scales_f16; /* out: [out][in/group] */
  uint16_t* zeros_f16;  /* out: [out][in/group] */
  float* losses;        /* out: [n_grid] */
  int32_t* best_idx;    /* out: [1] */
  float* s_best;        /* out: [in] */
  float* mean_abs;      /* out: [in], or NULL when not wanted */
} awq_layer_io;

/* Device bytes of the workspace awq_quantize_layers needs for layers of at
   most these sizes. Host-only. */
AWQ_API awq_status awq_pipeline_workspace_size(int64_t max_n_tok, int64_t max_out, int64_t max_in,
                                               int32_t w_dtype, const awq_config* cfg, size_t* bytes);

/* The whole method (statistics, alpha search, pack) for `count` layers
   whose inputs and outputs are in host memory, the way a model is quantised
   layer by layer. The workspace holds two slots of inputs and outputs: the
   search of layer i runs on `stream` while layer i+1's W and X are copied in
   and layer i-1's outputs are copied out on two library-owned copy streams,
   so the host link and the GPU work overlap. Results are the same as those
   of awq_act_stats, awq_search_layer and awq_quantize_pack called one layer
   at a time. Asynchronous: the outputs are in place once `stream` has
   passed this call (work queued on `stream` afterwards waits for the last
   copy). cfg->w_bit 2, 4 or 8 (packed as by awq_quantize_pack). ws: device, awq_pipeline_workspace_size()
   bytes for the largest layer dimensions; its first 4 bytes are the status
   word, which keeps the first device-side error of any layer (read it with
   awq_get_device_status). Calls from several host threads are serialised
   while they enqueue. */
AWQ_API awq_status awq_quantize_layers(const awq_layer_io* layers, int32_t count, int32_t w_dtype,
                                       const awq_config* cfg, void* ws, size_t ws_bytes, awq_stream_t stream);

/* ---------------------------------------------------------------- using the packed layer */

/* Largest token count, and token count times `in`, that awq_w4a16_gemv
   accepts (the tokens' activations are staged in one block's shared memory:
   as fp32 for groups of 32 and 64, 4.5 bytes per value with the bank
   padding; as bf16 pairs for groups of 128, 2.5 bytes per value). */
#define AWQ_W4A16_MAX_TOKENS 8
#define AWQ_W4A16_MAX_TOKEN_CHANNELS (44 * 1024)

/* The packed layer applied to a few tokens (w4a16, the decode case):
   y[t][r] = sum_k x[t][k] * (q[r][k] - z[r][g]) * scale[r][g], g = k / group,
   with q, scale, z as written by awq_quantize_pack ("AWQ: How
   Activation-Aware Quantization Saves 4-bit LLMs", "What do you actually
   deploy" and the decode remark after it: decoding is memory-bound and reads
   a quarter of the fp16 weight bytes). The codes quantise W * diag(s_best),
   so x is the layer input already divided by s_best (folded into its
   producer). x: device bf16 [n_tok][in] (x_dtype AWQ_BF16), 1 <= n_tok <=
   AWQ_W4A16_MAX_TOKENS and n_tok * in <= AWQ_W4A16_MAX_TOKEN_CHANNELS,
   else AWQ_ERR_UNSUPPORTED. qweight/scales_f16/zeros_f16: as
   awq_quantize_pack (qweight 16-byte aligned). y: device fp32 [n_tok][out].
   Each code is read once from memory, and every (q - z) is exact. Groups of
   32 and 64: fp32 products and fused multiply-adds in a fixed order. Groups
   of 128: tensor-core products of bf16 x with the exact (q - z), summed in
   fp32 per group, then scaled by the group's step in fp32 (when `in` / 128 is
   even and scales_f16 and zeros_f16 are 4-byte aligned, for two or more
   tokens, and for one token on a layer of at least 3 * 2^24 weights; otherwise
   the fp32 path). The order of every sum is fixed
   by the shapes and the device's SM count: repeated calls give the same
   bits. */
AWQ_API awq_status awq_w4a16_gemv(const void* x, int32_t x_dtype, int64_t n_tok, int64_t in,
                                  const int32_t* qweight, const uint16_t* scales_f16, const uint16_t* zeros_f16,
                                  int64_t out, const awq_config* cfg, float* y, awq_stream_t stream);

/* Bytes of the packed layer (codes + scales + zeros), host-only; 0 for
   invalid arguments. */
AWQ_API size_t awq_packed_bytes(int64_t out, int64_t in, const awq_config* cfg);

/* Synchronise `stream`, read the status word at the start of `ws` (device)
   into *status (host) and clear it. Returns AWQ_ERR_CUDA if the copy fails. */
AWQ_API awq_status awq_get_device_status(const void* ws, awq_stream_t stream, awq_status* status);

#ifdef __cplusplus
}
#endif

#endif /* AWQ_B300_H */
