// C ABI of the AWQ per-layer search and pack (declared in include/awq.h,
// include/awq_stages.h and include/awq_testing.h).
// Host code only: argument checks (all before any CUDA call), workspace
// carving, and the launch sequence of each step.
#include <string.h>

#include <algorithm>
#include <mutex>

#include "awq.h"
#include "awq_launch.h"
#include "awq_stages.h"
#include "awq_testing.h"
#include "awq_trace.h"

using namespace awq;

namespace {

constexpr size_t kAlign = 1024;

// Search size (flops of the alpha products) from which awq_search_layer
// runs the fake-quant as its own launch, followed by the single-CTA
// products, instead of the fused CTA-pair kernel. A search this long runs at
// the GPU's power limit, where the single-CTA products draw less energy per
// flop (70B-class layer, same box, back to back: 108 ms at 1.26 GHz and
// 0.85 kW against 135 ms at 0.95 GHz and 0.95 kW for the pair products).
constexpr double kLargeSearchFlops = AWQ_SEARCH_FUSED_MAX_FLOPS;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Flops of a search's alpha products: 2 * n_grid * n_tok * out * in.
inline double search_flops(int64_t n_tok, int64_t out, int64_t in, const awq_config& cfg) {
  return 2.0 * cfg.n_grid * (double)n_tok * (double)out * (double)in;
}
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor-core flops of the GRAM form: X^T X over the 128 x 256 tiles on and
// below the block diagonal, then per alpha the 128 x 256 tiles of every row
// block over their prefix of channel blocks.
double gram_flops(int64_t n_tok, int64_t out, int64_t in, const awq_config& cfg) {
  const int64_t ct = in / kTileM, m = ct / 2, b = ct % 2;
  const double h = 2.0 * (double)((m + 1) * (m + b)) * kTileM * kTileN * (double)gram_tokens_padded(n_tok);
  const int64_t nC = (in + kTileN - 1) / kTileN, nR = (out + kTileM - 1) / kTileM;
  double prefix = 0.0;
  for (int64_t c = 0; c < nC; ++c) prefix += (double)std::min<int64_t>(kTileN * (c + 1), in);
  return h + 2.0 * cfg.n_grid * (double)nR * kTileM * kTileN * prefix;
}

// Largest `in` of the GRAM form: the transpose's grid has in / 64 rows of
// tiles, at most 65535.
constexpr int64_t kGramMaxIn = (int64_t)65535 * 64;

// The form a search runs: AUTO resolves to GRAM when that form's flops are
// below 0.7 of the direct product's (the GRAM form adds X^T X, a transpose
// and a separate fake-quant launch), else to RESIDUAL.
int32_t resolve_form(int64_t n_tok, int64_t out, int64_t in, const awq_config& cfg) {
  if (cfg.loss_form != AWQ_LOSS_AUTO) return cfg.loss_form;
  if (in > kGramMaxIn) return AWQ_LOSS_RESIDUAL;
  return gram_flops(n_tok, out, in, cfg) < 0.7 * search_flops(n_tok, out, in, cfg) ? AWQ_LOSS_GRAM
                                                                                 : AWQ_LOSS_RESIDUAL;
}

// AWQ_ERR_UNSUPPORTED for a search whose form is GRAM beyond kGramMaxIn.
awq_status check_form(int64_t n_tok, int64_t out, int64_t in, const awq_config& cfg) {
  return resolve_form(n_tok, out, in, cfg) == AWQ_LOSS_GRAM && in > kGramMaxIn ? AWQ_ERR_UNSUPPORTED : AWQ_OK;
}

// The configuration a per-kernel stage call runs with: AUTO is RESIDUAL there.
awq_config stage_cfg(const awq_config* cfg) {
  awq_config c = *cfg;
  if (c.loss_form == AWQ_LOSS_AUTO) c.loss_form = AWQ_LOSS_RESIDUAL;
  return c;
}

// Largest sizes accepted: every index the kernels form stays below 2^31 per
// matrix dimension, and the TMA coordinates are 32-bit.
constexpr int64_t kMaxDim = (int64_t)1 << 30;

awq_status check_cfg(const awq_config* cfg) {
  if (cfg == nullptr) return AWQ_ERR_INVALID_ARG;
  if (cfg->n_grid < 1 || cfg->n_grid > kMaxGrid) return AWQ_ERR_INVALID_ARG;
  if (cfg->group <= 0 || cfg->w_bit <= 0) return AWQ_ERR_INVALID_ARG;
  if (!(cfg->sx_clamp_min > 0.0f) || !(cfg->delta_floor > 0.0f)) return AWQ_ERR_INVALID_ARG;
  if (cfg->loss_form < AWQ_LOSS_RESIDUAL || cfg->loss_form > AWQ_LOSS_AUTO) return AWQ_ERR_INVALID_ARG;
  if (cfg->zero_point != 0 && cfg->zero_point != 1) return AWQ_ERR_INVALID_ARG;
  // groups of 32, 64 or 128 weights (one or two groups per lane run of the
  // quantiser kernels); 2 to 8 bits per code in the search, whose codes are
  // never stored
  if (cfg->group != 32 && cfg->group != 64 && cfg->group != 128) return AWQ_ERR_UNSUPPORTED;
  if (cfg->w_bit < 2 || cfg->w_bit > 8) return AWQ_ERR_UNSUPPORTED;
  return AWQ_OK;
}

// The packed format holds codes of 2, 4 or 8 bits, 32/b to an int32.
awq_status check_packed_cfg(const awq_config* cfg) {
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  return (cfg->w_bit == 2 || cfg->w_bit == 4 || cfg->w_bit == 8) ? AWQ_OK : AWQ_ERR_UNSUPPORTED;
}

// The products over the packed layer read 4-bit codes.
awq_status check_product_cfg(const awq_config* cfg) {
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  return cfg->w_bit == 4 ? AWQ_OK : AWQ_ERR_UNSUPPORTED;
}

awq_status check_dims(int64_t n_tok, int64_t out, int64_t in) {
  if (n_tok < 1 || out < 1 || in < 1) return AWQ_ERR_INVALID_ARG;
  if (n_tok > kMaxDim || out > kMaxDim || in > kMaxDim) return AWQ_ERR_INVALID_ARG;
  if (in % kBlockCols != 0) return AWQ_ERR_INVALID_ARG;
  if (out * in > ((int64_t)1 << 40)) return AWQ_ERR_INVALID_ARG;
  return AWQ_OK;
}

awq_status check_wdtype(int32_t w_dtype) {
  if (w_dtype == AWQ_BF16 || w_dtype == AWQ_FP32) return AWQ_OK;
  return AWQ_ERR_INVALID_ARG;
}

awq_status check_xdtype(int32_t x_dtype) {
  if (x_dtype == AWQ_BF16) return AWQ_OK;
  if (x_dtype == AWQ_FP32) return AWQ_ERR_UNSUPPORTED;
  return AWQ_ERR_INVALID_ARG;
}

awq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? AWQ_OK : AWQ_ERR_CUDA; }

struct SearchLayout {
  size_t status, s, inv_s, op, partials, ready, row_acc, gram_h, total;
  int64_t mt, nt;
  int64_t per_alpha;  // partial sums per alpha
};

SearchLayout search_layout(int64_t n_tok, int64_t out, int64_t in, const awq_config& cfg_in) {
  awq_config cfg = cfg_in;
  cfg.loss_form = resolve_form(n_tok, out, in, cfg_in);
  SearchLayout L;
  const int64_t G = cfg.n_grid;
  const int64_t slots = cfg.loss_form == AWQ_LOSS_REFERENCE ? G + 1 : G;
  L.mt = (n_tok + kTileM - 1) / kTileM;
  L.nt = (out + kTileN - 1) / kTileN;
  size_t off = 0;
  L.status = off;
  off = align_up(off + 256, kAlign);
  L.s = off;
  off = align_up(off + (size_t)G * in * 4, kAlign);
  L.inv_s = off;
  off = align_up(off + (size_t)G * in * 4, kAlign);
  const bool gram = cfg.loss_form == AWQ_LOSS_GRAM;
  // GRAM form: X^T (bf16 [in][n_pad]) lives in the operand's space until the fake-quant writes it
  size_t op_bytes = (size_t)slots * out * in * 2;
  if (gram && (size_t)gram_tokens_padded(n_tok) * in * 2 > op_bytes) op_bytes = (size_t)gram_tokens_padded(n_tok) * in * 2;
  L.op = off;
  off = align_up(off + op_bytes, kAlign);
  L.per_alpha = gram ? gram_partials_per_alpha(out, in) : L.mt * L.nt * 4;
  L.partials = off;
  off = align_up(off + (size_t)G * L.per_alpha * 4, kAlign);
  L.ready = off;
  off = align_up(off + fused_ready_words(G, L.nt) * 4, kAlign);
  L.row_acc = off;  // fp64 [G][out], used when per-row losses are asked for
  off = align_up(off + (size_t)G * out * 8, kAlign);
  L.gram_h = off;  // GRAM form: bf16 [in][in]
  if (gram) off = align_up(off + (size_t)in * in * 2, kAlign);
  L.total = off;
  return L;
}

awq_status run_search(const void* W, int32_t w_dtype, int64_t out, int64_t in, const void* X, int64_t n_tok,
                      const float* mean_abs, const awq_config& c, float* losses, int32_t* best_idx, float* s_best,
                      uint8_t* base, const SearchLayout& L, cudaStream_t s, bool clear_status = true,
                      float* row_losses = nullptr);


// ------------------------------------------------------------- host-buffer layer pipeline
//
// Layers whose weights and activations sit in host memory go through two
// device slots: layer i's statistics, search and pack run on the caller's
// stream in slot i % 2 while layer i+1's inputs are copied into the other
// slot on a copy-in stream and layer i-1's outputs are copied out of it on
// a copy-out stream (the link is full duplex). Events order each slot's
// copy-in after the previous copy-out of that slot (which follows its
// compute), the compute after the copy-in, and the copy-out after the
// compute. The search workspace and the statistics scratch are shared by
// all layers, which run one after another on the caller's stream.

struct PipeLayout {
  size_t search, stats;  // offsets: search workspace (status word first), statistics scratch
  size_t slot[2];        // offsets of the two slots
  size_t W, X, mean_abs, qweight, scales, zeros, losses, best, s_best;  // offsets inside a slot
  size_t total;
};

// Bytes of search workspace that hold a search of any shape within the given
// maxima. Every region of a form's layout grows with each dimension; AUTO
// resolves per shape, so a smaller layer may take the other form than the
// maxima would: the bound is the larger of the two forms' layouts.
size_t search_bytes_bound(int64_t n_tok, int64_t out, int64_t in, const awq_config& cfg) {
  if (cfg.loss_form != AWQ_LOSS_AUTO) return search_layout(n_tok, out, in, cfg).total;
  awq_config r = cfg, g = cfg;
  r.loss_form = AWQ_LOSS_RESIDUAL;
  g.loss_form = AWQ_LOSS_GRAM;
  // AUTO takes the GRAM form only up to kGramMaxIn channels
  return std::max(search_layout(n_tok, out, in, r).total,
                  search_layout(n_tok, out, std::min(in, kGramMaxIn), g).total);
}

PipeLayout pipe_layout(int64_t n_tok, int64_t out, int64_t in, int32_t w_dtype, const awq_config& cfg) {
  PipeLayout P;
  const size_t wbytes = w_dtype == AWQ_BF16 ? 2 : 4;
  size_t off = 0;
  P.search = off;
  off = align_up(off + search_bytes_bound(n_tok, out, in, cfg), kAlign);
  P.stats = off;
  size_t stats_bytes = 0;
  awq_act_stats_workspace_size(n_tok, in, &stats_bytes);
  off = align_up(off + stats_bytes, kAlign);
  size_t o = 0;
  P.W = o;
  o = align_up(o + (size_t)out * in * wbytes, kAlign);
  P.X = o;
  o = align_up(o + (size_t)n_tok * in * 2, kAlign);
  P.mean_abs = o;
  o = align_up(o + (size_t)in * 4, kAlign);
  P.qweight = o;
  o = align_up(o + (size_t)out * in * cfg.w_bit / 8, kAlign);
  P.scales = o;
  o = align_up(o + (size_t)out * (in / cfg.group) * 2, kAlign);
  P.zeros = o;
  o = align_up(o + (size_t)out * (in / cfg.group) * 2, kAlign);
  P.losses = o;
  o = align_up(o + (size_t)cfg.n_grid * 4, kAlign);
  P.best = o;
  o = align_up(o + 4, kAlign);
  P.s_best = o;
  o = align_up(o + (size_t)in * 4, kAlign);
  P.slot[0] = off;
  P.slot[1] = off + o;
  P.total = off + 2 * o;
  return P;
}

// Copy streams and events of the pipeline, created once per device. The
// mutex is held while a call enqueues its work, so two host threads never
// interleave their event records on the shared streams.
struct PipeRes {
  bool ready = false;
  cudaStream_t in_s = nullptr, out_s = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t in_ev[2] = {}, comp_ev[2] = {}, out_ev[2] = {};
};
constexpr int kPipeDevices = 64;
std::mutex g_pipe_mu;
PipeRes g_pipe[kPipeDevices];

cudaError_t pipe_resources(int dev, PipeRes** out) {
  if (dev < 0 || dev >= kPipeDevices) return cudaErrorInvalidDevice;
  PipeRes& r = g_pipe[dev];
  if (!r.ready) {
    cudaError_t e = cudaStreamCreateWithFlags(&r.in_s, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&r.out_s, cudaStreamNonBlocking);
    cudaEvent_t* evs[8] = {&r.start, &r.done, &r.in_ev[0], &r.in_ev[1], &r.comp_ev[0], &r.comp_ev[1],
                           &r.out_ev[0], &r.out_ev[1]};
    for (int i = 0; i < 8 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
    r.ready = true;
  }
  *out = &r;
  return cudaSuccess;
}

awq_status check_layer_io(const awq_layer_io& L, const awq_config& cfg) {
  if (L.W == nullptr || L.X == nullptr || L.qweight == nullptr || L.scales_f16 == nullptr ||
      L.zeros_f16 == nullptr || L.losses == nullptr || L.best_idx == nullptr || L.s_best == nullptr)
    return AWQ_ERR_INVALID_ARG;
  awq_status st = check_dims(L.n_tok, L.out, L.in);
  if (st != AWQ_OK) return st;
  if (L.in % cfg.group != 0) return AWQ_ERR_INVALID_ARG;
  return AWQ_OK;
}

}  // namespace

extern "C" {

void awq_config_default(awq_config* cfg) {
  if (cfg == nullptr) return;
  cfg->w_bit = 4;
  cfg->group = 128;
  cfg->n_grid = 20;
  cfg->zero_point = 1;
  cfg->normalize = 1;
  cfg->sx_clamp_min = 1e-4f;
  cfg->delta_floor = 1e-5f;
  cfg->loss_form = AWQ_LOSS_AUTO;
  cfg->wait_timeout_ms = 0;
}

const char* awq_status_string(int status) {
  switch (status) {
    case AWQ_OK: return "ok";
    case AWQ_ERR_INVALID_ARG: return "invalid argument";
    case AWQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case AWQ_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case AWQ_ERR_WORKSPACE: return "workspace too small";
    case AWQ_ERR_CUDA: return "CUDA runtime error";
    case AWQ_ERR_TIMEOUT: return "device wait timed out";
    case AWQ_ERR_NONFINITE: return "non-finite loss";
    default: return "unknown status";
  }
}

// Statistics scratch: fp32 partial sums [chunks][in], then the per-strip tickets.
size_t stats_ticket_offset(int64_t n_tok, int64_t in) {
  return align_up((size_t)stats_chunks(n_tok, in) * (size_t)in * 4, kAlign);
}

awq_status awq_act_stats_workspace_size(int64_t n_tok, int64_t in, size_t* bytes) {
  if (bytes == nullptr || n_tok < 1 || in < 1 || n_tok > kMaxDim || in > kMaxDim) return AWQ_ERR_INVALID_ARG;
  *bytes = stats_ticket_offset(n_tok, in) + align_up((size_t)stats_strips(in) * 4, kAlign);
  return AWQ_OK;
}

awq_status awq_act_stats(const void* X, int32_t x_dtype, int64_t n_tok, int64_t in, float* mean_abs, void* ws,
                         size_t ws_bytes, awq_stream_t stream) {
  AWQ_TRACE("awq_act_stats");
  if (X == nullptr || mean_abs == nullptr || ws == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_xdtype(x_dtype);
  if (st != AWQ_OK) return st;
  if (n_tok < 1 || in < 1 || n_tok > kMaxDim || in > kMaxDim || in % 8 != 0) return AWQ_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(mean_abs) || !aligned16(ws)) return AWQ_ERR_MISALIGNED;
  size_t need = 0;
  awq_act_stats_workspace_size(n_tok, in, &need);
  if (ws_bytes < need) return AWQ_ERR_WORKSPACE;
  uint32_t* tickets = (uint32_t*)((uint8_t*)ws + stats_ticket_offset(n_tok, in));
  return from_cuda(launch_stats((const uint16_t*)X, n_tok, in, (float*)ws, tickets, mean_abs, (cudaStream_t)stream));
}

awq_status awq_workspace_size(int64_t n_tok, int64_t out, int64_t in, const awq_config* cfg, size_t* bytes) {
  if (bytes == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_dims(n_tok, out, in);
  if (st != AWQ_OK) return st;
  st = check_form(n_tok, out, in, *cfg);
  if (st != AWQ_OK) return st;
  *bytes = search_layout(n_tok, out, in, *cfg).total;
  return AWQ_OK;
}

awq_status awq_search_form(int64_t n_tok, int64_t out, int64_t in, const awq_config* cfg, int32_t* form) {
  if (form == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_dims(n_tok, out, in);
  if (st != AWQ_OK) return st;
  st = check_form(n_tok, out, in, *cfg);
  if (st != AWQ_OK) return st;
  *form = resolve_form(n_tok, out, in, *cfg);
  return AWQ_OK;
}

awq_status awq_search_tiles(int64_t n_tok, int64_t out, const awq_config* cfg, int64_t* m_tiles,
                            int64_t* n_tiles, int32_t* tile_m, int32_t* tile_n) {
  if (m_tiles == nullptr || n_tiles == nullptr || tile_m == nullptr || tile_n == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  if (n_tok < 1 || out < 1 || n_tok > kMaxDim || out > kMaxDim) return AWQ_ERR_INVALID_ARG;
  *m_tiles = (n_tok + kTileM - 1) / kTileM;
  *n_tiles = (out + kTileN - 1) / kTileN;
  *tile_m = kTileM;
  *tile_n = kTileN;
  return AWQ_OK;
}

awq_status awq_alpha_scales(const float* mean_abs, int64_t in, const awq_config* cfg, float* s, float* inv_s,
                            awq_stream_t stream) {
  AWQ_TRACE("awq_alpha_scales");
  if (mean_abs == nullptr || s == nullptr || inv_s == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  if (in < 1 || in > kMaxDim || in % kBlockCols != 0) return AWQ_ERR_INVALID_ARG;
  if (!aligned16(mean_abs) || !aligned16(s) || !aligned16(inv_s)) return AWQ_ERR_MISALIGNED;
  return from_cuda(launch_alpha_scales(mean_abs, in, *cfg, s, inv_s, (cudaStream_t)stream));
}

awq_status awq_fakequant(const void* W, int32_t w_dtype, int64_t out, int64_t in, const float* s,
                         const float* inv_s, const awq_config* cfg, uint16_t* op, awq_stream_t stream) {
  AWQ_TRACE("awq_fakequant");
  if (W == nullptr || s == nullptr || inv_s == nullptr || op == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_wdtype(w_dtype);
  if (st != AWQ_OK) return st;
  st = check_dims(1, out, in);
  if (st != AWQ_OK) return st;
  if (!aligned16(W) || !aligned16(s) || !aligned16(inv_s) || !aligned16(op)) return AWQ_ERR_MISALIGNED;
  return from_cuda(launch_fakequant(W, w_dtype, out, in, s, inv_s, *cfg, op, (cudaStream_t)stream));
}

awq_status awq_search_gemm(const void* X, int64_t n_tok, int64_t in, const uint16_t* op, int64_t out,
                           const awq_config* cfg, float* partials, uint32_t* status, awq_stream_t stream) {
  AWQ_TRACE("awq_search_gemm");
  if (X == nullptr || op == nullptr || partials == nullptr || status == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_dims(n_tok, out, in);
  if (st != AWQ_OK) return st;
  if (!aligned16(X) || !aligned16(op) || !aligned16(partials) || !aligned16(status)) return AWQ_ERR_MISALIGNED;
  // the products awq_search_layer runs for a search of this size
  const int single_cta = search_flops(n_tok, out, in, *cfg) >= kLargeSearchFlops ? 1 : 0;
  return from_cuda(launch_search_gemm((const uint16_t*)X, n_tok, in, op, out, *cfg, partials, status,
                                      (cudaStream_t)stream, nullptr, 0, single_cta));
}

awq_status awq_search_fused(const void* W, int32_t w_dtype, int64_t out, int64_t in, const void* X, int64_t n_tok,
                            const float* s, const float* inv_s, const awq_config* cfg, uint16_t* op, float* partials,
                            uint32_t* ready, uint32_t* status, awq_stream_t stream) {
  AWQ_TRACE("awq_search_fused");
  if (W == nullptr || X == nullptr || s == nullptr || inv_s == nullptr || op == nullptr || partials == nullptr ||
      ready == nullptr || status == nullptr)
    return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  const awq_config c = stage_cfg(cfg);
  if (c.loss_form != AWQ_LOSS_RESIDUAL) return AWQ_ERR_UNSUPPORTED;
  st = check_wdtype(w_dtype);
  if (st != AWQ_OK) return st;
  st = check_dims(n_tok, out, in);
  if (st != AWQ_OK) return st;
  if (!aligned16(W) || !aligned16(X) || !aligned16(s) || !aligned16(inv_s) || !aligned16(op) ||
      !aligned16(partials) || !aligned16(ready) || !aligned16(status))
    return AWQ_ERR_MISALIGNED;
  return from_cuda(launch_search_fused(W, w_dtype, (const uint16_t*)X, n_tok, in, s, inv_s, out, c, op, partials,
                                       ready, status, (cudaStream_t)stream));
}

awq_status awq_search_fused_withhold_unit(const void* W, int32_t w_dtype, int64_t out, int64_t in, const void* X,
                                          int64_t n_tok, const float* s, const float* inv_s, const awq_config* cfg,
                                          uint16_t* op, float* partials, uint32_t* ready, uint32_t* status,
                                          awq_stream_t stream) {
  AWQ_TRACE("awq_search_fused_withhold_unit");
  if (W == nullptr || X == nullptr || s == nullptr || inv_s == nullptr || op == nullptr || partials == nullptr ||
      ready == nullptr || status == nullptr)
    return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  const awq_config c = stage_cfg(cfg);
  if (c.loss_form != AWQ_LOSS_RESIDUAL) return AWQ_ERR_UNSUPPORTED;
  st = check_wdtype(w_dtype);
  if (st != AWQ_OK) return st;
  st = check_dims(n_tok, out, in);
  if (st != AWQ_OK) return st;
  if (!aligned16(W) || !aligned16(X) || !aligned16(s) || !aligned16(inv_s) || !aligned16(op) ||
      !aligned16(partials) || !aligned16(ready) || !aligned16(status))
    return AWQ_ERR_MISALIGNED;
  return from_cuda(launch_search_fused(W, w_dtype, (const uint16_t*)X, n_tok, in, s, inv_s, out, c, op, partials,
                                       ready, status, (cudaStream_t)stream, nullptr, 0));
}

awq_status awq_search_gemm_dump(const void* X, int64_t n_tok, int64_t in, const uint16_t* op, int64_t out,
                                const awq_config* cfg, float* partials, uint32_t* status, float* dump,
                                int32_t single_cta, awq_stream_t stream) {
  AWQ_TRACE("awq_search_gemm_dump");
  if (single_cta != 0 && single_cta != 1) return AWQ_ERR_INVALID_ARG;
  if (cfg != nullptr && cfg->loss_form != AWQ_LOSS_RESIDUAL && cfg->loss_form != AWQ_LOSS_AUTO)
    return AWQ_ERR_UNSUPPORTED;
  if (X == nullptr || op == nullptr || partials == nullptr || status == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_dims(n_tok, out, in);
  if (st != AWQ_OK) return st;
  if (!aligned16(X) || !aligned16(op) || !aligned16(partials) || !aligned16(status) || !aligned16(dump))
    return AWQ_ERR_MISALIGNED;
  return from_cuda(launch_search_gemm((const uint16_t*)X, n_tok, in, op, out, *cfg, partials, status,
                                      (cudaStream_t)stream, dump, 0, single_cta));
}

awq_status awq_gram_loss_withhold_fill(const uint16_t* op, int64_t out, int64_t in, const uint16_t* H,
                                       const awq_config* cfg, float* partials, uint32_t* status,
                                       awq_stream_t stream) {
  AWQ_TRACE("awq_gram_loss_withhold_fill");
  if (op == nullptr || H == nullptr || partials == nullptr || status == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_dims(1, out, in);
  if (st != AWQ_OK) return st;
  if (!aligned16(op) || !aligned16(H) || !aligned16(partials) || !aligned16(status)) return AWQ_ERR_MISALIGNED;
  return from_cuda(launch_gram_loss(op, out, in, *cfg, H, partials, status, (cudaStream_t)stream, nullptr, 1));
}

awq_status awq_search_gemm_withhold_fill(const void* X, int64_t n_tok, int64_t in, const uint16_t* op,
                                         int64_t out, const awq_config* cfg, float* partials, uint32_t* status,
                                         awq_stream_t stream) {
  AWQ_TRACE("awq_search_gemm_withhold_fill");
  if (X == nullptr || op == nullptr || partials == nullptr || status == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_dims(n_tok, out, in);
  if (st != AWQ_OK) return st;
  if (!aligned16(X) || !aligned16(op) || !aligned16(partials) || !aligned16(status)) return AWQ_ERR_MISALIGNED;
  return from_cuda(launch_search_gemm((const uint16_t*)X, n_tok, in, op, out, *cfg, partials, status,
                                      (cudaStream_t)stream, nullptr, 1));
}

awq_status awq_loss_select(const float* partials, int64_t n_tok, int64_t out, int64_t in, const float* s,
                           const awq_config* cfg, float* losses, int32_t* best_idx, float* s_best,
                           uint32_t* status, awq_stream_t stream) {
  AWQ_TRACE("awq_loss_select");
  if (partials == nullptr || s == nullptr || losses == nullptr || best_idx == nullptr || s_best == nullptr ||
      status == nullptr)
    return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_dims(n_tok, out, in);
  if (st != AWQ_OK) return st;
  if (!aligned16(partials) || !aligned16(s) || !aligned16(s_best)) return AWQ_ERR_MISALIGNED;
  const int64_t mt = (n_tok + kTileM - 1) / kTileM, nt = (out + kTileN - 1) / kTileN;
  const int64_t per_alpha = cfg->loss_form == AWQ_LOSS_GRAM ? gram_partials_per_alpha(out, in) : mt * nt * 4;
  return from_cuda(launch_loss_select(partials, cfg->n_grid, per_alpha, n_tok, out, s, in, losses, best_idx,
                                      s_best, status, (cudaStream_t)stream));
}

awq_status awq_gram_sizes(int64_t n_tok, int64_t out, int64_t in, int64_t* xt_elems, int64_t* h_elems,
                          int64_t* partials_per_alpha) {
  if (xt_elems == nullptr || h_elems == nullptr || partials_per_alpha == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_dims(n_tok, out, in);
  if (st != AWQ_OK) return st;
  *xt_elems = gram_tokens_padded(n_tok) * in;
  *h_elems = in * in;
  *partials_per_alpha = gram_partials_per_alpha(out, in);
  return AWQ_OK;
}

awq_status awq_gram_matrix(const void* X, int64_t n_tok, int64_t in, uint16_t* xt, uint16_t* H,
                           const awq_config* cfg, uint32_t* status, awq_stream_t stream) {
  AWQ_TRACE("awq_gram_matrix");
  if (X == nullptr || xt == nullptr || H == nullptr || status == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_dims(n_tok, 1, in);
  if (st != AWQ_OK) return st;
  if (in > kGramMaxIn) return AWQ_ERR_UNSUPPORTED;
  if (!aligned16(X) || !aligned16(xt) || !aligned16(H) || !aligned16(status)) return AWQ_ERR_MISALIGNED;
  return from_cuda(launch_gram_matrix((const uint16_t*)X, n_tok, in, xt, H, status, cfg->wait_timeout_ms,
                                      (cudaStream_t)stream));
}

awq_status awq_gram_loss(const uint16_t* op, int64_t out, int64_t in, const uint16_t* H, const awq_config* cfg,
                         float* partials, uint32_t* status, awq_stream_t stream) {
  AWQ_TRACE("awq_gram_loss");
  if (op == nullptr || H == nullptr || partials == nullptr || status == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_dims(1, out, in);
  if (st != AWQ_OK) return st;
  if (!aligned16(op) || !aligned16(H) || !aligned16(partials) || !aligned16(status)) return AWQ_ERR_MISALIGNED;
  return from_cuda(launch_gram_loss(op, out, in, *cfg, H, partials, status, (cudaStream_t)stream));
}

awq_status awq_search_layer(const void* W, int32_t w_dtype, int64_t out, int64_t in, const void* X,
                            int32_t x_dtype, int64_t n_tok, const float* mean_abs, const awq_config* cfg,
                            float* losses, int32_t* best_idx, float* s_best, float* row_losses, void* ws,
                            size_t ws_bytes, awq_stream_t stream) {
  AWQ_TRACE("awq_search_layer");
  if (W == nullptr || X == nullptr || mean_abs == nullptr || losses == nullptr || best_idx == nullptr ||
      s_best == nullptr || ws == nullptr)
    return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_wdtype(w_dtype);
  if (st != AWQ_OK) return st;
  st = check_xdtype(x_dtype);
  if (st != AWQ_OK) return st;
  st = check_dims(n_tok, out, in);
  if (st != AWQ_OK) return st;
  if (!aligned16(W) || !aligned16(X) || !aligned16(mean_abs) || !aligned16(s_best) || !aligned16(ws))
    return AWQ_ERR_MISALIGNED;
  st = check_form(n_tok, out, in, *cfg);
  if (st != AWQ_OK) return st;
  const SearchLayout L = search_layout(n_tok, out, in, *cfg);
  if (ws_bytes < L.total) return AWQ_ERR_WORKSPACE;

  if (row_losses != nullptr && (reinterpret_cast<uintptr_t>(row_losses) & 3u)) return AWQ_ERR_MISALIGNED;
  return run_search(W, w_dtype, out, in, X, n_tok, mean_abs, *cfg, losses, best_idx, s_best, (uint8_t*)ws, L,
                    (cudaStream_t)stream, true, row_losses);
}

awq_status awq_search_block_workspace_size(int64_t n_tok, const int64_t* outs, int32_t count, int64_t in,
                                           int32_t w_dtype, const awq_config* cfg, size_t* bytes) {
  if (bytes == nullptr || outs == nullptr || count < 1 || count > AWQ_BLOCK_MAX_LINEARS) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_wdtype(w_dtype);
  if (st != AWQ_OK) return st;
  int64_t total = 0;
  for (int i = 0; i < count; ++i) {
    if (outs[i] < 1) return AWQ_ERR_INVALID_ARG;
    total += outs[i];
  }
  st = check_dims(n_tok, total, in);
  if (st != AWQ_OK) return st;
  st = check_form(n_tok, total, in, *cfg);
  if (st != AWQ_OK) return st;
  const size_t wbytes = w_dtype == AWQ_BF16 ? 2 : 4;
  *bytes = search_layout(n_tok, total, in, *cfg).total + align_up((size_t)total * in * wbytes, kAlign);
  return AWQ_OK;
}

awq_status awq_search_block(const void* const* W_list, int32_t w_dtype, const int64_t* outs, int32_t count,
                            int64_t in, const void* X, int32_t x_dtype, int64_t n_tok, const float* mean_abs,
                            const awq_config* cfg, float* losses, int32_t* best_idx, float* s_best, void* ws,
                            size_t ws_bytes, awq_stream_t stream) {
  AWQ_TRACE("awq_search_block");
  if (W_list == nullptr || X == nullptr || mean_abs == nullptr || losses == nullptr || best_idx == nullptr ||
      s_best == nullptr || ws == nullptr)
    return AWQ_ERR_INVALID_ARG;
  size_t need = 0;
  awq_status st = awq_search_block_workspace_size(n_tok, outs, count, in, w_dtype, cfg, &need);
  if (st != AWQ_OK) return st;
  st = check_xdtype(x_dtype);
  if (st != AWQ_OK) return st;
  for (int i = 0; i < count; ++i) {
    if (W_list[i] == nullptr) return AWQ_ERR_INVALID_ARG;
    if (!aligned16(W_list[i])) return AWQ_ERR_MISALIGNED;
  }
  if (!aligned16(X) || !aligned16(mean_abs) || !aligned16(s_best) || !aligned16(ws)) return AWQ_ERR_MISALIGNED;
  if (ws_bytes < need) return AWQ_ERR_WORKSPACE;
  int64_t total = 0;
  for (int i = 0; i < count; ++i) total += outs[i];
  const SearchLayout L = search_layout(n_tok, total, in, *cfg);
  // the linears' rows, one after another, behind the search's own scratch
  uint8_t* base = (uint8_t*)ws;
  uint8_t* wcat = base + L.total;
  const size_t wbytes = w_dtype == AWQ_BF16 ? 2 : 4;
  cudaStream_t s = (cudaStream_t)stream;
  size_t off = 0;
  for (int i = 0; i < count; ++i) {
    const size_t b = (size_t)outs[i] * in * wbytes;
    if (cudaMemcpyAsync(wcat + off, W_list[i], b, cudaMemcpyDeviceToDevice, s) != cudaSuccess) return AWQ_ERR_CUDA;
    off += b;
  }
  return run_search(wcat, w_dtype, total, in, X, n_tok, mean_abs, *cfg, losses, best_idx, s_best, base, L, s);
}

}  // extern "C"

namespace {

awq_status run_search(const void* W, int32_t w_dtype, int64_t out, int64_t in, const void* X, int64_t n_tok,
                      const float* mean_abs, const awq_config& c, float* losses, int32_t* best_idx, float* s_best,
                      uint8_t* base, const SearchLayout& L, cudaStream_t s, bool clear_status,
                      float* row_losses) {
  awq_config resolved = c;
  resolved.loss_form = resolve_form(n_tok, out, in, c);
  const awq_config* cfg = &resolved;
  uint32_t* status = (uint32_t*)(base + L.status);
  float* sc = (float*)(base + L.s);
  float* inv = (float*)(base + L.inv_s);
  uint16_t* op = (uint16_t*)(base + L.op);
  float* partials = (float*)(base + L.partials);

  uint32_t* ready = (uint32_t*)(base + L.ready);
  double* row_acc = row_losses != nullptr ? (double*)(base + L.row_acc) : nullptr;

  cudaError_t e = clear_status ? cudaMemsetAsync(status, 0, 4, s) : cudaSuccess;
  if (e == cudaSuccess && row_acc != nullptr) e = cudaMemsetAsync(row_acc, 0, (size_t)cfg->n_grid * out * 8, s);
  if (e == cudaSuccess) e = launch_alpha_scales(mean_abs, in, *cfg, sc, inv, s);
  const double flops = search_flops(n_tok, out, in, *cfg);
  if (cfg->loss_form == AWQ_LOSS_GRAM) {
    // X^T X once (X^T in the operand's space), then the fake-quant, then the alphas' products against it
    uint16_t* H = (uint16_t*)(base + L.gram_h);
    if (e == cudaSuccess) e = launch_gram_matrix((const uint16_t*)X, n_tok, in, op, H, status, cfg->wait_timeout_ms, s);
    if (e == cudaSuccess) e = launch_fakequant(W, w_dtype, out, in, sc, inv, *cfg, op, s);
    if (e == cudaSuccess) e = launch_gram_loss(op, out, in, *cfg, H, partials, status, s, row_acc);
  } else if (cfg->loss_form == AWQ_LOSS_RESIDUAL && flops < kLargeSearchFlops) {
    // fake-quant runs inside the search kernel, ahead of the products that consume it
    if (e == cudaSuccess)
      e = launch_search_fused(W, w_dtype, (const uint16_t*)X, n_tok, in, sc, inv, out, *cfg, op, partials, ready,
                              status, s, nullptr, -1, row_acc);
  } else if (cfg->loss_form == AWQ_LOSS_RESIDUAL) {
    // the fake-quant launch, then the single-CTA products
    if (e == cudaSuccess) e = launch_fakequant(W, w_dtype, out, in, sc, inv, *cfg, op, s);
    if (e == cudaSuccess)
      e = launch_search_gemm((const uint16_t*)X, n_tok, in, op, out, *cfg, partials, status, s, nullptr, 0, 1, row_acc);
  } else {
    if (e == cudaSuccess) e = launch_fakequant(W, w_dtype, out, in, sc, inv, *cfg, op, s);
    if (e == cudaSuccess)
      e = launch_search_gemm((const uint16_t*)X, n_tok, in, op, out, *cfg, partials, status, s, nullptr, 0, 1, row_acc);
  }
  if (e == cudaSuccess)
    e = launch_loss_select(partials, cfg->n_grid, L.per_alpha, n_tok, out, sc, in, losses, best_idx, s_best, status,
                           s);
  if (e == cudaSuccess && row_acc != nullptr) e = launch_row_losses(row_acc, cfg->n_grid, out, n_tok, row_losses, s);
  return from_cuda(e);
}

}  // namespace

extern "C" {

awq_status awq_quantize_pack(const void* W, int32_t w_dtype, int64_t out, int64_t in, const float* s,
                             const awq_config* cfg, int32_t* qweight, uint16_t* scales_f16, uint16_t* zeros_f16,
                             awq_stream_t stream) {
  AWQ_TRACE("awq_quantize_pack");
  if (W == nullptr || s == nullptr || qweight == nullptr || scales_f16 == nullptr || zeros_f16 == nullptr)
    return AWQ_ERR_INVALID_ARG;
  awq_status st = check_packed_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_wdtype(w_dtype);
  if (st != AWQ_OK) return st;
  st = check_dims(1, out, in);
  if (st != AWQ_OK) return st;
  if (!aligned16(W) || !aligned16(s) || !aligned16(qweight)) return AWQ_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(scales_f16) & 1u) || (reinterpret_cast<uintptr_t>(zeros_f16) & 1u))
    return AWQ_ERR_MISALIGNED;
  return from_cuda(launch_pack(W, w_dtype, out, in, s, *cfg, qweight, scales_f16, zeros_f16,
                               (cudaStream_t)stream));
}

awq_status awq_w4a16_gemv(const void* x, int32_t x_dtype, int64_t n_tok, int64_t in, const int32_t* qweight,
                          const uint16_t* scales_f16, const uint16_t* zeros_f16, int64_t out, const awq_config* cfg,
                          float* y, awq_stream_t stream) {
  AWQ_TRACE("awq_w4a16_gemv");
  if (x == nullptr || qweight == nullptr || scales_f16 == nullptr || zeros_f16 == nullptr || y == nullptr)
    return AWQ_ERR_INVALID_ARG;
  awq_status st = check_product_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_xdtype(x_dtype);
  if (st != AWQ_OK) return st;
  st = check_dims(n_tok, out, in);
  if (st != AWQ_OK) return st;
  if (n_tok > AWQ_W4A16_MAX_TOKENS || n_tok * in > AWQ_W4A16_MAX_TOKEN_CHANNELS) return AWQ_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(qweight) || (reinterpret_cast<uintptr_t>(scales_f16) & 1u) ||
      (reinterpret_cast<uintptr_t>(zeros_f16) & 1u) || (reinterpret_cast<uintptr_t>(y) & 3u))
    return AWQ_ERR_MISALIGNED;
  return from_cuda(launch_w4a16_gemv((const uint16_t*)x, n_tok, in, qweight, scales_f16, zeros_f16, out,
                                     cfg->group, y, (cudaStream_t)stream));
}

// Prefill product scratch: status word, the product's tile partials, then the bf16 weight.
struct GemmLayout {
  size_t status, partials, w_hat, total;
};

GemmLayout gemm_layout(int64_t n_tok, int64_t out, int64_t in) {
  GemmLayout L;
  const int64_t mt = (n_tok + kTileM - 1) / kTileM, nt = (out + kTileN - 1) / kTileN;
  L.status = 0;
  L.partials = kAlign;
  L.w_hat = align_up(L.partials + (size_t)mt * nt * 4 * 4, kAlign);
  L.total = align_up(L.w_hat + (size_t)out * in * 2, kAlign);
  return L;
}

awq_status awq_w4a16_gemm_workspace_size(int64_t n_tok, int64_t in, int64_t out, const awq_config* cfg,
                                         size_t* bytes) {
  if (bytes == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_product_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_dims(n_tok, out, in);
  if (st != AWQ_OK) return st;
  *bytes = gemm_layout(n_tok, out, in).total;
  return AWQ_OK;
}

awq_status awq_w4a16_gemm(const void* x, int32_t x_dtype, int64_t n_tok, int64_t in, const int32_t* qweight,
                          const uint16_t* scales_f16, const uint16_t* zeros_f16, int64_t out, const awq_config* cfg,
                          float* y, void* ws, size_t ws_bytes, awq_stream_t stream) {
  AWQ_TRACE("awq_w4a16_gemm");
  if (x == nullptr || qweight == nullptr || scales_f16 == nullptr || zeros_f16 == nullptr || y == nullptr ||
      ws == nullptr)
    return AWQ_ERR_INVALID_ARG;
  awq_status st = check_product_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_xdtype(x_dtype);
  if (st != AWQ_OK) return st;
  st = check_dims(n_tok, out, in);
  if (st != AWQ_OK) return st;
  if (!aligned16(x) || !aligned16(qweight) || !aligned16(y) || !aligned16(ws) ||
      (reinterpret_cast<uintptr_t>(scales_f16) & 1u) || (reinterpret_cast<uintptr_t>(zeros_f16) & 1u))
    return AWQ_ERR_MISALIGNED;
  const GemmLayout L = gemm_layout(n_tok, out, in);
  if (ws_bytes < L.total) return AWQ_ERR_WORKSPACE;
  uint8_t* base = (uint8_t*)ws;
  uint16_t* w_hat = (uint16_t*)(base + L.w_hat);
  uint32_t* status = (uint32_t*)(base + L.status);
  const cudaStream_t s = (cudaStream_t)stream;
  awq_config one = *cfg;  // the product of one operand: the search kernels with a grid of one alpha
  one.n_grid = 1;
  one.loss_form = AWQ_LOSS_RESIDUAL;
  cudaError_t e = cudaMemsetAsync(status, 0, 4, s);
  if (e == cudaSuccess) e = launch_w4_expand(qweight, scales_f16, zeros_f16, out, in, cfg->group, w_hat, s);
  if (e == cudaSuccess)
    e = launch_search_gemm((const uint16_t*)x, n_tok, in, w_hat, out, one, (float*)(base + L.partials), status, s, y);
  return from_cuda(e);
}

size_t awq_packed_bytes(int64_t out, int64_t in, const awq_config* cfg) {
  if (check_cfg(cfg) != AWQ_OK || out < 1 || in < 1 || in % cfg->group != 0) return 0;
  const size_t n = (size_t)out * (size_t)in;
  const size_t codes = n * (size_t)cfg->w_bit / 8;
  const size_t groups = n / (size_t)cfg->group;
  return codes + groups * 2 + (cfg->zero_point ? groups * 2 : 0);
}

awq_status awq_get_device_status(const void* ws, awq_stream_t stream, awq_status* status) {
  if (ws == nullptr || status == nullptr) return AWQ_ERR_INVALID_ARG;
  uint32_t word = 0;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(&word, ws, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(const_cast<void*>(ws), 0, 4, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return AWQ_ERR_CUDA;
  *status = (awq_status)word;
  return AWQ_OK;
}

awq_status awq_pipeline_workspace_size(int64_t max_n_tok, int64_t max_out, int64_t max_in, int32_t w_dtype,
                                       const awq_config* cfg, size_t* bytes) {
  if (bytes == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_packed_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_wdtype(w_dtype);
  if (st != AWQ_OK) return st;
  st = check_dims(max_n_tok, max_out, max_in);
  if (st != AWQ_OK) return st;
  if (cfg->loss_form == AWQ_LOSS_GRAM && max_in > kGramMaxIn) return AWQ_ERR_UNSUPPORTED;
  *bytes = pipe_layout(max_n_tok, max_out, max_in, w_dtype, *cfg).total;
  return AWQ_OK;
}

awq_status awq_quantize_layers(const awq_layer_io* layers, int32_t count, int32_t w_dtype, const awq_config* cfg,
                               void* ws, size_t ws_bytes, awq_stream_t stream) {
  AWQ_TRACE("awq_quantize_layers");
  if (layers == nullptr || count < 1 || ws == nullptr) return AWQ_ERR_INVALID_ARG;
  awq_status st = check_packed_cfg(cfg);
  if (st != AWQ_OK) return st;
  st = check_wdtype(w_dtype);
  if (st != AWQ_OK) return st;
  if (!aligned16(ws)) return AWQ_ERR_MISALIGNED;
  int64_t n_max = 1, out_max = 1, in_max = 1;
  for (int32_t i = 0; i < count; ++i) {
    st = check_layer_io(layers[i], *cfg);
    if (st != AWQ_OK) return st;
    n_max = layers[i].n_tok > n_max ? layers[i].n_tok : n_max;
    out_max = layers[i].out > out_max ? layers[i].out : out_max;
    in_max = layers[i].in > in_max ? layers[i].in : in_max;
  }
  // every region of the layout grows with each dimension, so the layout of
  // the largest dimensions holds every layer at the same offsets (for the
  // search region, whichever loss form each layer resolves to)
  const PipeLayout P = pipe_layout(n_max, out_max, in_max, w_dtype, *cfg);
  if (ws_bytes < P.total) return AWQ_ERR_WORKSPACE;
  for (int32_t i = 0; i < count; ++i) {  // checked before anything is queued
    st = check_form(layers[i].n_tok, layers[i].out, layers[i].in, *cfg);
    if (st != AWQ_OK) return st;
    if (search_layout(layers[i].n_tok, layers[i].out, layers[i].in, *cfg).total > P.stats - P.search)
      return AWQ_ERR_WORKSPACE;  // holds by construction
  }

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return AWQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  PipeRes* R = nullptr;
  if (pipe_resources(dev, &R) != cudaSuccess) return AWQ_ERR_CUDA;
  const cudaStream_t cs = (cudaStream_t)stream;
  uint8_t* base = (uint8_t*)ws;
  const size_t wbytes = w_dtype == AWQ_BF16 ? 2 : 4;
  // the copy streams start after the work already queued on the caller's
  // stream (which may still use this workspace); the status word is
  // cleared once, so it keeps the first error of any layer
  cudaError_t e = cudaMemsetAsync(base + P.search, 0, 4, cs);
  if (e == cudaSuccess) e = cudaEventRecord(R->start, cs);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(R->in_s, R->start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(R->out_s, R->start, 0);
  for (int32_t i = 0; i < count && e == cudaSuccess; ++i) {
    const awq_layer_io& L = layers[i];
    const int b = i & 1;
    uint8_t* slot = base + P.slot[b];
    const size_t gcols = (size_t)(L.in / cfg->group);
    // copy-in: after the previous copy-out of this slot (two layers back)
    if (i >= 2) e = cudaStreamWaitEvent(R->in_s, R->out_ev[b], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(slot + P.W, L.W, (size_t)L.out * L.in * wbytes, cudaMemcpyDefault, R->in_s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(slot + P.X, L.X, (size_t)L.n_tok * L.in * 2, cudaMemcpyDefault, R->in_s);
    if (e == cudaSuccess) e = cudaEventRecord(R->in_ev[b], R->in_s);
    // compute on the caller's stream
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, R->in_ev[b], 0);
    float* mean_abs = (float*)(slot + P.mean_abs);
    float* s_best = (float*)(slot + P.s_best);
    if (e == cudaSuccess) {
      uint8_t* sws = base + P.stats;
      e = launch_stats((const uint16_t*)(slot + P.X), L.n_tok, L.in, (float*)sws,
                       (uint32_t*)(sws + stats_ticket_offset(L.n_tok, L.in)), mean_abs, cs);
    }
    if (e == cudaSuccess) {
      const SearchLayout SL = search_layout(L.n_tok, L.out, L.in, *cfg);
      st = run_search(slot + P.W, w_dtype, L.out, L.in, slot + P.X, L.n_tok, mean_abs, *cfg,
                      (float*)(slot + P.losses), (int32_t*)(slot + P.best), s_best, base + P.search, SL, cs,
                      /*clear_status=*/false);
      if (st != AWQ_OK) return st;
    }
    if (e == cudaSuccess)
      e = launch_pack(slot + P.W, w_dtype, L.out, L.in, s_best, *cfg, (int32_t*)(slot + P.qweight),
                      (uint16_t*)(slot + P.scales), (uint16_t*)(slot + P.zeros), cs);
    if (e == cudaSuccess) e = cudaEventRecord(R->comp_ev[b], cs);
    // copy-out
    if (e == cudaSuccess) e = cudaStreamWaitEvent(R->out_s, R->comp_ev[b], 0);
    const struct {
      void* dst;
      size_t off, bytes;
    } outs[6] = {{L.qweight, P.qweight, (size_t)L.out * L.in * cfg->w_bit / 8},
                 {L.scales_f16, P.scales, (size_t)L.out * gcols * 2},
                 {L.zeros_f16, P.zeros, (size_t)L.out * gcols * 2},
                 {L.losses, P.losses, (size_t)cfg->n_grid * 4},
                 {L.best_idx, P.best, 4},
                 {L.s_best, P.s_best, (size_t)L.in * 4}};
    for (int k = 0; k < 6 && e == cudaSuccess; ++k)
      e = cudaMemcpyAsync(outs[k].dst, slot + outs[k].off, outs[k].bytes, cudaMemcpyDefault, R->out_s);
    if (e == cudaSuccess && L.mean_abs != nullptr)
      e = cudaMemcpyAsync(L.mean_abs, mean_abs, (size_t)L.in * 4, cudaMemcpyDefault, R->out_s);
    if (e == cudaSuccess) e = cudaEventRecord(R->out_ev[b], R->out_s);
  }
  // the caller's stream continues once the last outputs have arrived
  if (e == cudaSuccess) e = cudaEventRecord(R->done, R->out_s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, R->done, 0);
  return from_cuda(e);
}

awq_status awq_bounds_report(uint64_t* failures, int32_t* unit, uint64_t* line, uint64_t* offset) {
  if (failures == nullptr || unit == nullptr || line == nullptr || offset == nullptr) return AWQ_ERR_INVALID_ARG;
#ifdef AWQ_CHECKED
  cudaError_t (*const take[4])(unsigned long long*) = {take_oob_kernels, take_oob_search, take_oob_w4a16,
                                                       take_oob_gram};
  *failures = 0;
  *unit = 0;
  *line = 0;
  *offset = 0;
  for (int u = 0; u < 4; ++u) {
    unsigned long long rec[3] = {0, 0, 0};
    if (take[u](rec) != cudaSuccess) return AWQ_ERR_CUDA;
    if (rec[0] != 0 && *unit == 0) {
      *unit = u + 1;
      *line = rec[1];
      *offset = rec[2];
    }
    *failures += rec[0];
  }
  return AWQ_OK;
#else
  return AWQ_ERR_UNSUPPORTED;
#endif
}

awq_status awq_bounds_selftest(float* buf, int32_t n, awq_stream_t stream) {
  if (buf == nullptr || n < 1) return AWQ_ERR_INVALID_ARG;
#ifdef AWQ_CHECKED
  return from_cuda(launch_bounds_selftest(buf, n, (cudaStream_t)stream));
#else
  (void)stream;
  return AWQ_ERR_UNSUPPORTED;
#endif
}

}  // extern "C"
