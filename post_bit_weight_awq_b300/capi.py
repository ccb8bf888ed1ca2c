"""ctypes binding of libawq.so, one Python function per C entry point.

Argument marshalling only: tensors are passed as raw device pointers with
their sizes; every step of the computation runs in the library's CUDA kernels.
There is no fallback: if libawq.so cannot be loaded, importing the binding's
functions raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

# AWQ_LIBRARY selects another build of the library (libawq_checked.so, the bounds-checked kernels).
LIB_PATH = os.environ.get("AWQ_LIBRARY") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "libawq.so")

AWQ_OK = 0
AWQ_ERR_INVALID_ARG = 1
AWQ_ERR_UNSUPPORTED = 2
AWQ_ERR_MISALIGNED = 3
AWQ_ERR_WORKSPACE = 4
AWQ_ERR_CUDA = 5
AWQ_ERR_TIMEOUT = 6
AWQ_ERR_NONFINITE = 7

AWQ_BF16 = 0
AWQ_FP32 = 1

AWQ_LOSS_RESIDUAL = 0
AWQ_LOSS_REFERENCE = 1
AWQ_LOSS_GRAM = 2
AWQ_LOSS_AUTO = 3

# limits of include/awq.h
AWQ_W4A16_MAX_TOKENS = 8
AWQ_W4A16_MAX_TOKEN_CHANNELS = 44 * 1024
AWQ_BLOCK_MAX_LINEARS = 16

# Every function that include/awq.h (the product interface) declares.
EXPORTED = (
    "awq_config_default",
    "awq_status_string",
    "awq_act_stats_workspace_size",
    "awq_act_stats",
    "awq_act_stats_noalloc",
    "awq_workspace_size",
    "awq_search_form",
    "awq_search_layer",
    "awq_search_block_workspace_size",
    "awq_search_block",
    "awq_quantize_pack",
    "awq_w4a16_gemv",
    "awq_w4a16_gemm_workspace_size",
    "awq_w4a16_gemm",
    "awq_pipeline_workspace_size",
    "awq_quantize_layers",
    "awq_packed_bytes",
    "awq_get_device_status",
)


class AwqConfig(ctypes.Structure):
    _fields_ = [
        ("w_bit", ctypes.c_int32),
        ("group", ctypes.c_int32),
        ("n_grid", ctypes.c_int32),
        ("zero_point", ctypes.c_int32),
        ("normalize", ctypes.c_int32),
        ("sx_clamp_min", ctypes.c_float),
        ("delta_floor", ctypes.c_float),
        ("loss_form", ctypes.c_int32),
        ("wait_timeout_ms", ctypes.c_uint32),
    ]


class AwqLayerIO(ctypes.Structure):
    """One layer of awq_quantize_layers (host or device pointers)."""
    _fields_ = [
        ("W", ctypes.c_void_p),
        ("X", ctypes.c_void_p),
        ("n_tok", ctypes.c_int64),
        ("out", ctypes.c_int64),
        ("in_", ctypes.c_int64),
        ("qweight", ctypes.c_void_p),
        ("scales_f16", ctypes.c_void_p),
        ("zeros_f16", ctypes.c_void_p),
        ("losses", ctypes.c_void_p),
        ("best_idx", ctypes.c_void_p),
        ("s_best", ctypes.c_void_p),
        ("mean_abs", ctypes.c_void_p),
    ]


class AwqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t
_CFG = ctypes.POINTER(AwqConfig)


def lib() -> ctypes.CDLL:
    """Load libawq.so (built in-tree by ``post_bit_weight_awq_b300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libawq.so is not built ({LIB_PATH}); run python -m post_bit_weight_awq_b300.build")
    L = ctypes.CDLL(LIB_PATH)
    sig = {
        "awq_config_default": (None, [_CFG]),
        "awq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "awq_act_stats_workspace_size": (ctypes.c_int, [_I64, _I64, ctypes.POINTER(_SZ)]),
        "awq_act_stats": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _P, _SZ, _P]),
        "awq_act_stats_noalloc": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _P]),
        "awq_workspace_size": (ctypes.c_int, [_I64, _I64, _I64, _CFG, ctypes.POINTER(_SZ)]),
        "awq_search_form": (ctypes.c_int, [_I64, _I64, _I64, _CFG, ctypes.POINTER(_I32)]),
        "awq_search_layer": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _I32, _I64, _P, _CFG, _P, _P, _P, _P, _P, _SZ,
                                            _P]),
        "awq_search_block_workspace_size": (ctypes.c_int, [_I64, _P, _I32, _I64, _I32, _CFG, ctypes.POINTER(_SZ)]),
        "awq_search_block": (ctypes.c_int, [_P, _I32, _P, _I32, _I64, _P, _I32, _I64, _P, _CFG, _P, _P, _P, _P, _SZ,
                                            _P]),
        "awq_quantize_pack": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _CFG, _P, _P, _P, _P]),
        "awq_w4a16_gemv": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _P, _P, _I64, _CFG, _P, _P]),
        "awq_w4a16_gemm_workspace_size": (ctypes.c_int, [_I64, _I64, _I64, _CFG, ctypes.POINTER(_SZ)]),
        "awq_w4a16_gemm": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _P, _P, _I64, _CFG, _P, _P, _SZ, _P]),
        "awq_pipeline_workspace_size": (ctypes.c_int, [_I64, _I64, _I64, _I32, _CFG, ctypes.POINTER(_SZ)]),
        "awq_quantize_layers": (ctypes.c_int, [_P, _I32, _I32, _CFG, _P, _SZ, _P]),
        "awq_packed_bytes": (_SZ, [_I64, _I64, _CFG]),
        "awq_get_device_status": (ctypes.c_int, [_P, _P, ctypes.POINTER(ctypes.c_int)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().awq_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != AWQ_OK:
        raise AwqError(status, where)


def config(**kw) -> AwqConfig:
    """Default configuration (4 bits, groups of 128, 20 alphas, zero point,
    normalised scales, AUTO loss form) with fields overridden by ``kw``."""
    c = AwqConfig()
    lib().awq_config_default(ctypes.byref(c))
    for k, v in kw.items():
        if not hasattr(c, k):
            raise AttributeError(k)
        setattr(c, k, v)
    return c


# ----------------------------------------------------------------- marshalling


def _ptr(t) -> Optional[int]:
    """Device pointer of a tensor (or a raw int pointer, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return AWQ_BF16
    if t.dtype == torch.float32:
        return AWQ_FP32
    return 99  # rejected by the library as AWQ_ERR_INVALID_ARG


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


# ----------------------------------------------------------------- size queries


def awq_act_stats_workspace_size(n_tok: int, in_features: int) -> int:
    b = _SZ(0)
    _check(lib().awq_act_stats_workspace_size(n_tok, in_features, ctypes.byref(b)), "awq_act_stats_workspace_size")
    return b.value


def awq_workspace_size(n_tok: int, out_features: int, in_features: int, cfg: AwqConfig) -> int:
    b = _SZ(0)
    _check(lib().awq_workspace_size(n_tok, out_features, in_features, ctypes.byref(cfg), ctypes.byref(b)),
           "awq_workspace_size")
    return b.value


def awq_search_form(n_tok: int, out_features: int, in_features: int, cfg: AwqConfig) -> int:
    """The loss form awq_search_layer runs for this shape (AUTO resolved)."""
    f = _I32(0)
    _check(lib().awq_search_form(n_tok, out_features, in_features, ctypes.byref(cfg), ctypes.byref(f)),
           "awq_search_form")
    return f.value




def awq_packed_bytes(out_features: int, in_features: int, cfg: AwqConfig) -> int:
    return int(lib().awq_packed_bytes(out_features, in_features, ctypes.byref(cfg)))


# ----------------------------------------------------------------- compute calls


def awq_act_stats(X, mean_abs, ws, stream=None, *, n_tok=None, in_features=None, x_dtype=None,
                  ws_bytes=None) -> None:
    n = X.shape[0] if n_tok is None else n_tok
    k = X.shape[1] if in_features is None else in_features
    xd = _dtype_code(X) if x_dtype is None else x_dtype
    wb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check(lib().awq_act_stats(_ptr(X), xd, n, k, _ptr(mean_abs), _ptr(ws), wb, _stream(stream)), "awq_act_stats")


def awq_act_stats_noalloc(X, mean_abs, stream=None, *, n_tok=None, in_features=None, x_dtype=None) -> None:
    """awq_act_stats without caller scratch, for callers that cannot allocate
    (library-owned fixed array; see include/awq.h for its size limit and the
    rule that overlapping calls race)."""
    n = X.shape[0] if n_tok is None else n_tok
    k = X.shape[1] if in_features is None else in_features
    xd = _dtype_code(X) if x_dtype is None else x_dtype
    _check(lib().awq_act_stats_noalloc(_ptr(X), xd, n, k, _ptr(mean_abs), _stream(stream)), "awq_act_stats_noalloc")


def awq_search_layer(W, X, mean_abs, cfg: AwqConfig, losses, best_idx, s_best, ws, stream=None, *,
                     out_features=None, in_features=None, n_tok=None, w_dtype=None, x_dtype=None,
                     ws_bytes=None, row_losses=None) -> None:
    N = W.shape[0] if out_features is None else out_features
    K = W.shape[1] if in_features is None else in_features
    n = X.shape[0] if n_tok is None else n_tok
    wd = _dtype_code(W) if w_dtype is None else w_dtype
    xd = _dtype_code(X) if x_dtype is None else x_dtype
    wb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check(lib().awq_search_layer(_ptr(W), wd, N, K, _ptr(X), xd, n, _ptr(mean_abs), ctypes.byref(cfg),
                                  _ptr(losses), _ptr(best_idx), _ptr(s_best), _ptr(row_losses), _ptr(ws), wb,
                                  _stream(stream)),
           "awq_search_layer")


def awq_search_block_workspace_size(n_tok: int, outs, in_features: int, cfg: AwqConfig, w_dtype: int = AWQ_BF16) -> int:
    arr = (ctypes.c_int64 * len(outs))(*outs)
    b = _SZ(0)
    _check(lib().awq_search_block_workspace_size(n_tok, ctypes.cast(arr, _P), len(outs), in_features, w_dtype,
                                                 ctypes.byref(cfg), ctypes.byref(b)), "awq_search_block_workspace_size")
    return b.value


def awq_search_block(Ws, X, mean_abs, cfg: AwqConfig, losses, best_idx, s_best, ws, stream=None, *, outs=None,
                     in_features=None, n_tok=None, w_dtype=None, x_dtype=None, ws_bytes=None) -> None:
    """Ws: sequence of device weight tensors [out_j, in] (or raw pointers with ``outs``)."""
    outs = [W.shape[0] for W in Ws] if outs is None else list(outs)
    K = Ws[0].shape[1] if in_features is None else in_features
    n = X.shape[0] if n_tok is None else n_tok
    wd = _dtype_code(Ws[0]) if w_dtype is None else w_dtype
    xd = _dtype_code(X) if x_dtype is None else x_dtype
    wb = _nbytes(ws) if ws_bytes is None else ws_bytes
    ptrs = (ctypes.c_void_p * len(Ws))(*[_ptr(W) for W in Ws])
    arr = (ctypes.c_int64 * len(outs))(*outs)
    _check(lib().awq_search_block(ctypes.cast(ptrs, _P), wd, ctypes.cast(arr, _P), len(outs), K, _ptr(X), xd, n,
                                  _ptr(mean_abs), ctypes.byref(cfg), _ptr(losses), _ptr(best_idx), _ptr(s_best),
                                  _ptr(ws), wb, _stream(stream)), "awq_search_block")






def awq_pipeline_workspace_size(max_n_tok: int, max_out: int, max_in: int, w_dtype: int, cfg: AwqConfig) -> int:
    n = _SZ(0)
    _check(lib().awq_pipeline_workspace_size(max_n_tok, max_out, max_in, w_dtype, ctypes.byref(cfg),
                                             ctypes.byref(n)), "awq_pipeline_workspace_size")
    return n.value


def layer_io(W, X, qweight, scales, zeros, losses, best_idx, s_best, mean_abs=None, *, n_tok=None, out=None,
             in_features=None) -> AwqLayerIO:
    """An AwqLayerIO from tensors (host or device) or raw pointers with the sizes given."""
    return AwqLayerIO(_ptr(W), _ptr(X), X.shape[0] if n_tok is None else n_tok, W.shape[0] if out is None else out,
                      W.shape[1] if in_features is None else in_features, _ptr(qweight), _ptr(scales), _ptr(zeros),
                      _ptr(losses), _ptr(best_idx), _ptr(s_best), _ptr(mean_abs))


def awq_quantize_layers(layers, w_dtype: int, cfg: AwqConfig, ws, stream=None, *, ws_bytes=None) -> None:
    """layers: sequence of AwqLayerIO (see ``layer_io``)."""
    arr = (AwqLayerIO * len(layers))(*layers)
    wb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check(lib().awq_quantize_layers(ctypes.cast(arr, _P), len(layers), w_dtype, ctypes.byref(cfg), _ptr(ws), wb,
                                     _stream(stream)), "awq_quantize_layers")


def awq_quantize_pack(W, s, cfg: AwqConfig, qweight, scales, zeros, stream=None, *, out_features=None,
                      in_features=None, w_dtype=None) -> None:
    N = W.shape[0] if out_features is None else out_features
    K = W.shape[1] if in_features is None else in_features
    wd = _dtype_code(W) if w_dtype is None else w_dtype
    _check(lib().awq_quantize_pack(_ptr(W), wd, N, K, _ptr(s), ctypes.byref(cfg), _ptr(qweight), _ptr(scales),
                                   _ptr(zeros), _stream(stream)), "awq_quantize_pack")


def awq_w4a16_gemm_workspace_size(n_tok: int, in_features: int, out_features: int, cfg: AwqConfig) -> int:
    n = _SZ(0)
    _check(lib().awq_w4a16_gemm_workspace_size(n_tok, in_features, out_features, ctypes.byref(cfg), ctypes.byref(n)),
           "awq_w4a16_gemm_workspace_size")
    return n.value


def awq_w4a16_gemm(x, qweight, scales, zeros, cfg: AwqConfig, y, ws, stream=None, *, n_tok=None, in_features=None,
                   out_features=None, x_dtype=None, ws_bytes=None) -> None:
    """y [n_tok, out] fp32 = x [n_tok, in] bf16 times the packed layer's bf16 weight (prefill product)."""
    n = x.shape[0] if n_tok is None else n_tok
    K = x.shape[1] if in_features is None else in_features
    N = qweight.shape[0] if out_features is None else out_features
    xd = _dtype_code(x) if x_dtype is None else x_dtype
    wb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check(lib().awq_w4a16_gemm(_ptr(x), xd, n, K, _ptr(qweight), _ptr(scales), _ptr(zeros), N, ctypes.byref(cfg),
                                _ptr(y), _ptr(ws), wb, _stream(stream)), "awq_w4a16_gemm")


def awq_w4a16_gemv(x, qweight, scales, zeros, cfg: AwqConfig, y, stream=None, *, n_tok=None, in_features=None,
                   out_features=None, x_dtype=None) -> None:
    n = x.shape[0] if n_tok is None else n_tok
    K = x.shape[1] if in_features is None else in_features
    N = qweight.shape[0] if out_features is None else out_features
    xd = _dtype_code(x) if x_dtype is None else x_dtype
    _check(lib().awq_w4a16_gemv(_ptr(x), xd, n, K, _ptr(qweight), _ptr(scales), _ptr(zeros), N, ctypes.byref(cfg),
                                _ptr(y), _stream(stream)), "awq_w4a16_gemv")


def awq_get_device_status(ws, stream=None) -> int:
    st = ctypes.c_int(0)
    _check(lib().awq_get_device_status(_ptr(ws), _stream(stream), ctypes.byref(st)), "awq_get_device_status")
    return st.value
