"""ctypes binding of the stage entry points (include/awq_stages.h) and the
test aids (include/awq_testing.h) of libawq.so.

These calls are not the product interface (include/awq.h, bound in
``capi``): the stage calls run one kernel of the alpha search each, so that
the tests and the benchmark can check and time the kernels one by one, and
the test aids look inside the kernels or make a device-side wait run out on
purpose. Only the tests and the benchmark import this module. Argument
marshalling only, on the same loaded library as ``capi``.
"""
from __future__ import annotations

import ctypes

from . import capi
from .capi import (_CFG, _I32, _I64, _P, AwqConfig, _check, _dtype_code, _ptr, _stream)

# include/awq_stages.h: searches below this many product flops run the fused kernel in awq_search_layer.
AWQ_SEARCH_FUSED_MAX_FLOPS = 2e13

# Every function that include/awq_stages.h declares.
STAGE_EXPORTED = (
    "awq_alpha_scales",
    "awq_fakequant",
    "awq_search_tiles",
    "awq_search_gemm",
    "awq_search_fused",
    "awq_gram_sizes",
    "awq_gram_matrix",
    "awq_gram_loss",
    "awq_loss_select",
)

# Every function that include/awq_testing.h declares.
TESTING_EXPORTED = (
    "awq_search_gemm_dump",
    "awq_search_gemm_withhold_fill",
    "awq_search_fused_withhold_unit",
    "awq_gram_loss_withhold_fill",
    "awq_bounds_report",
    "awq_bounds_selftest",
)

_ready = False


def lib() -> ctypes.CDLL:
    """The library loaded by ``capi.lib()``, with the signatures of the stage
    calls and test aids set."""
    global _ready
    L = capi.lib()
    if _ready:
        return L
    sig = {
        "awq_alpha_scales": (ctypes.c_int, [_P, _I64, _CFG, _P, _P, _P]),
        "awq_fakequant": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _P, _CFG, _P, _P]),
        "awq_search_tiles": (ctypes.c_int, [_I64, _I64, _CFG, ctypes.POINTER(_I64), ctypes.POINTER(_I64),
                                            ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
        "awq_search_gemm": (ctypes.c_int, [_P, _I64, _I64, _P, _I64, _CFG, _P, _P, _P]),
        "awq_search_fused": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _I64, _P, _P, _CFG, _P, _P, _P, _P, _P]),
        "awq_gram_sizes": (ctypes.c_int, [_I64, _I64, _I64, ctypes.POINTER(_I64), ctypes.POINTER(_I64),
                                          ctypes.POINTER(_I64)]),
        "awq_gram_matrix": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _CFG, _P, _P]),
        "awq_gram_loss": (ctypes.c_int, [_P, _I64, _I64, _P, _CFG, _P, _P, _P]),
        "awq_loss_select": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _CFG, _P, _P, _P, _P, _P]),
        "awq_search_gemm_dump": (ctypes.c_int, [_P, _I64, _I64, _P, _I64, _CFG, _P, _P, _P, _I32, _P]),
        "awq_search_gemm_withhold_fill": (ctypes.c_int, [_P, _I64, _I64, _P, _I64, _CFG, _P, _P, _P]),
        "awq_search_fused_withhold_unit": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _I64, _P, _P, _CFG, _P, _P, _P,
                                                          _P, _P]),
        "awq_gram_loss_withhold_fill": (ctypes.c_int, [_P, _I64, _I64, _P, _CFG, _P, _P, _P]),
        "awq_bounds_report": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(_I32),
                                             ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]),
        "awq_bounds_selftest": (ctypes.c_int, [_P, _I32, _P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _ready = True
    return L


def awq_alpha_scales(mean_abs, cfg: AwqConfig, s, inv_s, stream=None, *, in_features=None) -> None:
    K = mean_abs.shape[0] if in_features is None else in_features
    _check(lib().awq_alpha_scales(_ptr(mean_abs), K, ctypes.byref(cfg), _ptr(s), _ptr(inv_s), _stream(stream)),
           "awq_alpha_scales")


def awq_fakequant(W, s, inv_s, cfg: AwqConfig, op, stream=None, *, out_features=None, in_features=None,
                  w_dtype=None) -> None:
    N = W.shape[0] if out_features is None else out_features
    K = W.shape[1] if in_features is None else in_features
    wd = _dtype_code(W) if w_dtype is None else w_dtype
    _check(lib().awq_fakequant(_ptr(W), wd, N, K, _ptr(s), _ptr(inv_s), ctypes.byref(cfg), _ptr(op),
                               _stream(stream)), "awq_fakequant")


def awq_search_tiles(n_tok: int, out_features: int, cfg: AwqConfig):
    mt, nt, tm, tn = _I64(0), _I64(0), _I32(0), _I32(0)
    _check(lib().awq_search_tiles(n_tok, out_features, ctypes.byref(cfg), ctypes.byref(mt), ctypes.byref(nt),
                                  ctypes.byref(tm), ctypes.byref(tn)), "awq_search_tiles")
    return mt.value, nt.value, tm.value, tn.value


def awq_search_gemm(X, op, cfg: AwqConfig, partials, status, stream=None, *, n_tok=None, in_features=None,
                    out_features=None) -> None:
    n = X.shape[0] if n_tok is None else n_tok
    K = X.shape[1] if in_features is None else in_features
    N = op.shape[-2] if out_features is None else out_features
    _check(lib().awq_search_gemm(_ptr(X), n, K, _ptr(op), N, ctypes.byref(cfg), _ptr(partials), _ptr(status),
                                 _stream(stream)), "awq_search_gemm")


def awq_search_fused(W, X, s, inv_s, cfg: AwqConfig, op, partials, ready, status, stream=None, *, out_features=None,
                     in_features=None, n_tok=None, w_dtype=None) -> None:
    N = W.shape[0] if out_features is None else out_features
    K = W.shape[1] if in_features is None else in_features
    n = X.shape[0] if n_tok is None else n_tok
    wd = _dtype_code(W) if w_dtype is None else w_dtype
    _check(lib().awq_search_fused(_ptr(W), wd, N, K, _ptr(X), n, _ptr(s), _ptr(inv_s), ctypes.byref(cfg), _ptr(op),
                                  _ptr(partials), _ptr(ready), _ptr(status), _stream(stream)), "awq_search_fused")


def awq_gram_sizes(n_tok: int, out_features: int, in_features: int):
    """(xt elements, H elements, partial sums per alpha) of the GRAM loss form."""
    xt, h, pa = _I64(0), _I64(0), _I64(0)
    _check(lib().awq_gram_sizes(n_tok, out_features, in_features, ctypes.byref(xt), ctypes.byref(h), ctypes.byref(pa)),
           "awq_gram_sizes")
    return xt.value, h.value, pa.value


def awq_gram_matrix(X, xt, H, cfg: AwqConfig, status, stream=None, *, n_tok=None, in_features=None) -> None:
    n = X.shape[0] if n_tok is None else n_tok
    K = X.shape[1] if in_features is None else in_features
    _check(lib().awq_gram_matrix(_ptr(X), n, K, _ptr(xt), _ptr(H), ctypes.byref(cfg), _ptr(status), _stream(stream)),
           "awq_gram_matrix")


def awq_gram_loss(op, H, cfg: AwqConfig, partials, status, stream=None, *, out_features=None,
                  in_features=None) -> None:
    N = op.shape[-2] if out_features is None else out_features
    K = op.shape[-1] if in_features is None else in_features
    _check(lib().awq_gram_loss(_ptr(op), N, K, _ptr(H), ctypes.byref(cfg), _ptr(partials), _ptr(status),
                               _stream(stream)), "awq_gram_loss")


def awq_loss_select(partials, s, cfg: AwqConfig, losses, best_idx, s_best, status, stream=None, *, n_tok,
                    out_features, in_features) -> None:
    _check(lib().awq_loss_select(_ptr(partials), n_tok, out_features, in_features, _ptr(s), ctypes.byref(cfg),
                                 _ptr(losses), _ptr(best_idx), _ptr(s_best), _ptr(status), _stream(stream)),
           "awq_loss_select")


def awq_search_gemm_dump(X, op, cfg: AwqConfig, partials, status, dump, stream=None, *, n_tok=None,
                         in_features=None, out_features=None, single_cta=0) -> None:
    n = X.shape[0] if n_tok is None else n_tok
    K = X.shape[1] if in_features is None else in_features
    N = op.shape[-2] if out_features is None else out_features
    _check(lib().awq_search_gemm_dump(_ptr(X), n, K, _ptr(op), N, ctypes.byref(cfg), _ptr(partials), _ptr(status),
                                      _ptr(dump), single_cta, _stream(stream)), "awq_search_gemm_dump")


def awq_search_gemm_withhold_fill(X, op, cfg: AwqConfig, partials, status, stream=None, *, n_tok=None,
                                  in_features=None, out_features=None) -> None:
    n = X.shape[0] if n_tok is None else n_tok
    K = X.shape[1] if in_features is None else in_features
    N = op.shape[-2] if out_features is None else out_features
    _check(lib().awq_search_gemm_withhold_fill(_ptr(X), n, K, _ptr(op), N, ctypes.byref(cfg), _ptr(partials),
                                               _ptr(status), _stream(stream)), "awq_search_gemm_withhold_fill")


def awq_search_fused_withhold_unit(W, X, s, inv_s, cfg: AwqConfig, op, partials, ready, status, stream=None, *,
                                   out_features=None, in_features=None, n_tok=None, w_dtype=None) -> None:
    N = W.shape[0] if out_features is None else out_features
    K = W.shape[1] if in_features is None else in_features
    n = X.shape[0] if n_tok is None else n_tok
    wd = _dtype_code(W) if w_dtype is None else w_dtype
    _check(lib().awq_search_fused_withhold_unit(_ptr(W), wd, N, K, _ptr(X), n, _ptr(s), _ptr(inv_s),
                                                ctypes.byref(cfg), _ptr(op), _ptr(partials), _ptr(ready),
                                                _ptr(status), _stream(stream)), "awq_search_fused_withhold_unit")


def awq_bounds_report():
    """(failed checks, source unit, line, offset) of a checked build; raises AwqError from a release build."""
    f, u, ln, off = ctypes.c_uint64(0), _I32(0), ctypes.c_uint64(0), ctypes.c_uint64(0)
    _check(lib().awq_bounds_report(ctypes.byref(f), ctypes.byref(u), ctypes.byref(ln), ctypes.byref(off)),
           "awq_bounds_report")
    return f.value, u.value, ln.value, off.value


def awq_bounds_selftest(buf, stream=None, *, n=None) -> None:
    _check(lib().awq_bounds_selftest(_ptr(buf), buf.numel() if n is None else n, _stream(stream)),
           "awq_bounds_selftest")


def awq_gram_loss_withhold_fill(op, H, cfg: AwqConfig, partials, status, stream=None, *, out_features=None,
                                in_features=None) -> None:
    N = op.shape[-2] if out_features is None else out_features
    K = op.shape[-1] if in_features is None else in_features
    _check(lib().awq_gram_loss_withhold_fill(_ptr(op), N, K, _ptr(H), ctypes.byref(cfg), _ptr(partials),
                                             _ptr(status), _stream(stream)), "awq_gram_loss_withhold_fill")
