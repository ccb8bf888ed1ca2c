"""CPU oracle for AWQ's per-layer activation-aware scale search and INT4 pack.

TEST INFRASTRUCTURE ONLY. This is a plain, slow, fp64 numpy statement of what
the library computes. Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import it; the CUDA path never does, and the
two share no code. Every input comes from the seeded generator in
``workloads``; nothing here reads a value produced by the CUDA path.

Sources (web pages on AWQ, cited by title and section):

* [AWQ-devto]  "AWQ: How Activation-Aware Quantization Saves 4-bit LLMs"
  - "How does AWQ decide which weights to protect?" (channel_importance listing)
  - "How does AWQ protect channels without mixed precision?" (search_scale
    listing and the two remarks after it)
  - "What do you actually deploy" (the quant_config listing: zero point on,
    group size 128, 4 bits)
* [AWQ-SWP]    "AWQ > Salient Weight Preservation": the step-size equation
  (range over 2^b - 1 levels) and the scaling equation (w*s times x/s).
* [AWQ-Sum]    "AWQ > Summary": "Salient weight identification" (mean absolute
  activation) and "The scaling formula" (the exponent alpha).
* [AWQ-Gloss]  "What is AWQ Quantization? Definition & 4-Bit Weight Compression
  in Enterprise AI", step "INT4 Weight Packing & Export" (4-bit codes held in
  INT32 containers).
* [AWQ-Ref]    "AWQ (Activation-Aware Weight Quantization) - AI Glossary",
  "Example: Where 4-bit memory saving comes from" (13e9-weight arithmetic).
* [AWQ-devto] "What do you actually deploy" (w4a16: 4-bit weights, 16-bit
  activations) and the decode remark after it (token-by-token decoding is
  memory-bound, so reading a quarter of the weight bytes is the payoff).

Readings taken where the pages are silent or disagree:

* Quantiser: asymmetric min/max with a zero point [AWQ-SWP step-size equation;
  AWQ-devto quant_config], not the symmetric max|w| form of [AWQ-devto, "Why
  does naive 4-bit quantization wreck LLM accuracy?"].
* Rounding is round-half-to-even; the zero point is rne(-vmin/delta), not
  clamped; codes are clamped to [0, 2^b - 1]; a constant group gets
  delta = max(delta, delta_floor).
* Codes are decided in fp32 ("pinned" quantiser): every arithmetic step is done
  in fp64 and rounded to the nearest fp32. For + - * / of fp32 operands this
  equals the correctly rounded fp32 operation (fp64 has 53 >= 2*24 + 2 bits,
  so the double rounding is innocuous), which is what the CUDA kernels use.
* Scale normalisation s /= sqrt(max(s)*min(s)) is not on the pages; the
  library applies it by specification. In exact arithmetic it leaves the
  dequantised weight unchanged (Q(c*V) = c*Q(V) for c > 0 when the floor is
  not hit); ``normalize=False`` turns it off.
* The clamp constant of the statistic is 1e-4 rounded to fp32 (CLAMP_MIN):
  the search_scale listing clamps a float tensor, where the constant takes
  the tensor's precision, and the library's parameter is an fp32 value.
* Grid alpha_i = i / n_grid for i = 0..n_grid-1 (0 .. 0.95 at 20 points), and
  the first strict minimum wins [AWQ-devto search_scale listing].
* Packing: 8 codes per 32-bit word along the input dimension, code k of a word
  in bits [4k, 4k+4), lowest column in the lowest nibble; scales and zeros are
  stored as fp16 (round-to-nearest-even), one of each per group.
"""
from __future__ import annotations

from typing import Callable, Dict, Optional

import numpy as np

__all__ = [
    "CLAMP_MIN",
    "f32",
    "bf16",
    "w4a16_expand_bf16",
    "channel_importance",
    "alpha_grid",
    "awq_scales",
    "quantize_groups",
    "dequantize_groups",
    "fake_quantize",
    "output_mse",
    "output_sq_err_sum",
    "search_scale",
    "search_scale_block",
    "pack_words",
    "unpack_words",
    "quantize_pack",
    "packed_bytes",
    "w4a16_linear",
]


CLAMP_MIN = float(np.float32(1e-4))


def f32(x) -> np.ndarray:
    """Round fp64 values to the nearest fp32 (ties to even); fp64 out."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def channel_importance(X) -> np.ndarray:
    """Mean absolute activation of each input channel over the tokens.

    [AWQ-devto, "How does AWQ decide which weights to protect?",
    channel_importance listing; AWQ-Sum, "Salient weight identification"]
    X: [n_tok, in]. Returns fp64 [in].
    """
    X = np.asarray(X, dtype=np.float64)
    return np.abs(X).mean(axis=0)


def alpha_grid(n_grid: int) -> np.ndarray:
    """alpha_i = i / n_grid, i = 0..n_grid-1 [AWQ-devto, search_scale listing]."""
    return np.array([i / n_grid for i in range(n_grid)], dtype=np.float64)


def awq_scales(sx, alpha: float, clamp_min: float = CLAMP_MIN, normalize: bool = True) -> np.ndarray:
    """Per-input-channel scale s = max(sx, clamp_min) ** alpha.

    [AWQ-devto, search_scale listing: clamp then power; AWQ-Sum, "The scaling
    formula": alpha sets how strongly high-activation channels are favoured.]
    With ``normalize`` the vector is divided by sqrt(max(s) * min(s)) (library
    specification, not on the pages).
    """
    base = np.maximum(np.asarray(sx, dtype=np.float64), clamp_min)
    s = base ** float(alpha)
    if normalize:
        s = s / np.sqrt(s.max() * s.min())
    return s


def quantize_groups(
    V,
    w_bit: int = 4,
    group: int = 128,
    delta_floor: float = 1e-5,
    pinned: bool = True,
    round_fn: Callable[[np.ndarray], np.ndarray] = np.rint,
    zero_point: bool = True,
):
    """Group-wise min/max quantisation of V [rows, in] along ``in``.

    Asymmetric, with a zero point (the default) [AWQ-SWP, step-size equation:
    delta = (v_max - v_min) / (2^b - 1); AWQ-devto quant_config: zero point
    on, groups of 128 along the input]. Per group:
    delta = max((vmax - vmin) / (2^b - 1), delta_floor),
    z = round(-vmin / delta), q = clamp(round(v / delta) + z, 0, 2^b - 1).
    Symmetric, ``zero_point=False`` [AWQ-devto, "Why does naive 4-bit
    quantization wreck LLM accuracy?": delta = max|w| / 2^(N-1),
    Q(w) = delta * round(w / delta)]: delta = max(max|v| / 2^(b-1),
    delta_floor); the rounded value lies in [-2^(b-1), 2^(b-1)] and is stored
    in b bits as q = clamp(round(v / delta) + 2^(b-1), 0, 2^b - 1), i.e. with
    the fixed zero point z = 2^(b-1) (the largest positive weight of a group
    clamps to 2^(b-1) - 1 steps).
    ``pinned`` rounds every step to fp32 (the precision the kernels decide
    codes in); ``pinned=False`` is the same formula in fp64. ``round_fn`` is
    round-half-to-even; a test may pass the identity to remove rounding.
    Returns (q [rows, in], delta [rows, in/group], z [rows, in/group]).
    """
    V = np.asarray(V, dtype=np.float64)
    rows, K = V.shape
    if K % group:
        raise ValueError("in_features must be a multiple of the group size")
    r = f32 if pinned else (lambda a: np.asarray(a, dtype=np.float64))
    qmax = float(2**w_bit - 1)
    Vg = V.reshape(rows, K // group, group)
    vmax = Vg.max(axis=2)
    vmin = Vg.min(axis=2)
    if zero_point:
        delta = r(r(vmax - vmin) / qmax)
        delta = np.maximum(delta, r(np.float64(delta_floor)))
        z = round_fn(r(-vmin / delta))
    else:
        half = float(2 ** (w_bit - 1))
        delta = r(np.maximum(-vmin, vmax) / half)  # max |v| / 2^(b-1)
        delta = np.maximum(delta, r(np.float64(delta_floor)))
        z = np.full_like(delta, half)
    q = np.clip(round_fn(r(Vg / delta[:, :, None])) + z[:, :, None], 0.0, qmax)
    return q.reshape(rows, K), delta, z


def dequantize_groups(q, delta, z, group: int = 128) -> np.ndarray:
    """(q - z) * delta per group, fp64."""
    q = np.asarray(q, dtype=np.float64)
    rows, K = q.shape
    qg = q.reshape(rows, K // group, group)
    return ((qg - z[:, :, None]) * delta[:, :, None]).reshape(rows, K)


def fake_quantize(
    W,
    s,
    w_bit: int = 4,
    group: int = 128,
    delta_floor: float = 1e-5,
    pinned: bool = True,
    round_fn: Callable[[np.ndarray], np.ndarray] = np.rint,
    zero_point: bool = True,
) -> np.ndarray:
    """W_hat = Q(W * s) / s: scale columns up, quantise, fold the scale back.

    [AWQ-devto, search_scale listing: weight columns times s, quantize_fn,
    then divide by s; AWQ-SWP scaling equation: w_ij*s_j times x_j/s_j keeps
    y_i unchanged, so Q(W*s)/s is the effective weight.]
    With ``pinned`` the scale is first rounded to fp32 and W*s is an fp32
    product, as the kernels form it; the fold-back is fp64.
    """
    W = np.asarray(W, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    if pinned:
        s = f32(s)
        V = f32(W * s[None, :])
    else:
        V = W * s[None, :]
    q, delta, z = quantize_groups(V, w_bit, group, delta_floor, pinned, round_fn, zero_point)
    return dequantize_groups(q, delta, z, group) / s[None, :]


def output_mse(X, W, W_hat) -> float:
    """mean((X W_hat^T - X W^T)^2) over tokens x outputs.

    [AWQ-devto, search_scale listing: reference output from the unquantised
    weight, then the squared error of the quantised layer's output, averaged.]
    """
    X = np.asarray(X, dtype=np.float64)
    y_ref = X @ np.asarray(W, dtype=np.float64).T
    y = X @ np.asarray(W_hat, dtype=np.float64).T
    return float(np.mean((y - y_ref) ** 2))


def output_sq_err_sum(X, W, W_hat) -> float:
    """sum((X (W_hat - W)^T)^2): the same error, as a sum, by distributivity.

    X W_hat^T - X W^T = X (W_hat - W)^T, so ``output_mse`` equals this sum over
    n_tok * out. It takes one product instead of two, which makes full-size
    layers affordable on the CPU; the tests pin the two forms together.
    """
    X = np.asarray(X, dtype=np.float64)
    E = np.asarray(W_hat, dtype=np.float64) - np.asarray(W, dtype=np.float64)
    D = X @ E.T
    return float(np.sum(D * D))


def search_scale(
    W,
    X,
    sx,
    n_grid: int = 20,
    clamp_min: float = CLAMP_MIN,
    normalize: bool = True,
    w_bit: int = 4,
    group: int = 128,
    delta_floor: float = 1e-5,
    pinned: bool = True,
    loss: Optional[Callable] = None,
    zero_point: bool = True,
) -> Dict[str, object]:
    """Grid search over alpha for the scale with the lowest output MSE.

    [AWQ-devto, "How does AWQ protect channels without mixed precision?",
    search_scale listing; AWQ-Sum, "Efficient algorithm": a per-layer grid
    search over the exponent.] The first strict minimum wins.
    Returns losses [n_grid], best_idx, best alpha, s_best (fp64) and all s.
    """
    loss = output_mse if loss is None else loss
    best_err, best_i = float("inf"), -1
    losses, scales = [], []
    for i, alpha in enumerate(alpha_grid(n_grid)):
        s = awq_scales(sx, alpha, clamp_min, normalize)
        W_hat = fake_quantize(W, s, w_bit, group, delta_floor, pinned, zero_point=zero_point)
        err = loss(X, W, W_hat)
        losses.append(err)
        scales.append(s)
        if err < best_err:
            best_err, best_i = err, i
    return {
        "losses": np.array(losses),
        "best_idx": best_i,
        "best_alpha": best_i / n_grid,
        "s_best": scales[best_i],
        "scales": np.stack(scales),
    }


def search_scale_block(W_list, X, sx, **kw) -> Dict[str, object]:
    """One scale for several linears that read the same X.

    [AWQ-SWP: the inverse scale is folded into the preceding LayerNorm /
    RMSNorm, so all linears fed by that norm (q/k/v, or gate/up) must share
    s.] The search scores each alpha by the output MSE of all of them
    together: the search of the layer whose weight is their rows stacked.
    """
    return search_scale(np.concatenate([np.asarray(W, dtype=np.float64) for W in W_list], axis=0), X, sx, **kw)


def pack_words(q, w_bit: int = 4) -> np.ndarray:
    """Pack b-bit codes [rows, in] into int32 words [rows, in * b / 32].

    [AWQ-Gloss, "INT4 Weight Packing & Export": 4-bit codes in INT32
    containers.] Code of column (32/b)*j + k goes to bits [b*k, b*k + b) of
    word j (for b = 4: column 8j+k in bits [4k, 4k+4)). b divides 32: 2, 4 or 8.
    """
    if w_bit not in (2, 4, 8):
        raise ValueError("codes are packed for 2, 4 or 8 bits")
    per = 32 // w_bit
    q = np.asarray(q)
    rows, K = q.shape
    if K % per:
        raise ValueError("in_features must be a multiple of the codes per word")
    qi = q.astype(np.int64).reshape(rows, K // per, per)
    if qi.min(initial=0) < 0 or qi.max(initial=0) > 2**w_bit - 1:
        raise ValueError("codes outside the range of the width")
    words = np.zeros((rows, K // per), dtype=np.int64)
    for k in range(per):
        words += qi[:, :, k] << (w_bit * k)
    return words.astype(np.uint32).view(np.int32)


def unpack_words(words, in_features: int, w_bit: int = 4) -> np.ndarray:
    """Inverse of ``pack_words``: int32 [rows, in*b/32] -> codes int64 [rows, in]."""
    per = 32 // w_bit
    w = np.asarray(words).view(np.uint32).astype(np.int64)
    rows = w.shape[0]
    out = np.zeros((rows, in_features // per, per), dtype=np.int64)
    for k in range(per):
        out[:, :, k] = (w >> (w_bit * k)) & (2**w_bit - 1)
    return out.reshape(rows, in_features)


def quantize_pack(W, s, w_bit: int = 4, group: int = 128, delta_floor: float = 1e-5, zero_point: bool = True):
    """Final codes of W * diag(s), packed, with fp16 group scales and zeros.

    [AWQ-Gloss, "INT4 Weight Packing & Export"; AWQ-Ref, memory example: one
    16-bit scale per group of 128; AWQ-devto quant_config: zero point on.]
    Codes use the pinned fp32 quantiser on fl32(W * fl32(s)); the stored scale
    is fp16(delta) and the stored zero fp16(z).
    Codes of 2 or 8 bits pack the same way, 16 or 4 to a word (3-bit codes do
    not fill a 32-bit word evenly and are not packed).
    Returns dict(qweight int32 [out, in*b/32], scales fp16, zeros fp16, codes,
    delta fp32-valued fp64, z).
    """
    if w_bit not in (2, 4, 8):
        raise ValueError("codes are packed for 2, 4 or 8 bits")
    W = np.asarray(W, dtype=np.float64)
    s32 = f32(np.asarray(s, dtype=np.float64))
    V = f32(W * s32[None, :])
    q, delta, z = quantize_groups(V, w_bit, group, delta_floor, pinned=True, zero_point=zero_point)
    # a zero point beyond the fp16 range (a near-constant group far from 0, step at the floor) rounds to inf,
    # as an IEEE round-to-nearest conversion does; that is the stored value, not an error
    with np.errstate(over="ignore"):
        zeros16 = z.astype(np.float32).astype(np.float16)
    return {
        "qweight": pack_words(q, w_bit),
        "scales": delta.astype(np.float32).astype(np.float16),
        "zeros": zeros16,
        "codes": q.astype(np.int64),
        "delta": delta,
        "z": z,
    }


def packed_bytes(out_features: int, in_features: int, group: int = 128, w_bit: int = 4,
                 zero_point: bool = True) -> Dict[str, int]:
    """Bytes of the packed layer: codes, fp16 scales, fp16 zeros.

    [AWQ-Ref, "Example: Where 4-bit memory saving comes from": half a byte per
    weight plus one 2-byte scale per group.]
    """
    n = out_features * in_features
    codes = n * w_bit // 8
    scales = (n // group) * 2
    zeros = (n // group) * 2 if zero_point else 0
    return {"codes": codes, "scales": scales, "zeros": zeros, "total": codes + scales + zeros}


def w4a16_linear(x, qweight, scales_f16, zeros_f16, group: int = 128) -> np.ndarray:
    """y = x @ W_hat^T for a packed layer: W_hat[r, k] = (q[r, k] - z[r, g]) * scale[r, g].

    [AWQ-devto, "What do you actually deploy": 4-bit weights with 16-bit
    activations; the decode remark: decoding reads the packed weights.]
    The layer is the output of ``quantize_pack``: codes of W * diag(s), so the
    caller passes activations already divided by s (the fold into the
    preceding norm described in "AWQ > Salient Weight Preservation").
    x: [M, in]; qweight int32 [out, in/8]; scales/zeros fp16 [out, in/group].
    fp64 arithmetic on the stored fp16 values. Returns fp64 [M, out].
    """
    x = np.asarray(x, dtype=np.float64)
    out_f = np.asarray(qweight).shape[0]
    K = np.asarray(qweight).shape[1] * 8
    q = unpack_words(qweight, K).astype(np.float64)
    sc = np.asarray(scales_f16, dtype=np.float16).astype(np.float64)
    z = np.asarray(zeros_f16, dtype=np.float16).astype(np.float64)
    W_hat = dequantize_groups(q, sc, z, group)
    assert W_hat.shape == (out_f, K)
    return x @ W_hat.T


def bf16(x) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even), via fp32, returned as fp64.

    The value is first rounded to fp32 (exact for the products below), then
    the low 16 bits of the fp32 pattern are rounded away half-to-even.
    """
    x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    b = x32.view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def w4a16_expand_bf16(qweight, scales_f16, zeros_f16, group: int = 128) -> np.ndarray:
    """The packed layer as the bf16 weight the prefill product multiplies:
    W_hat[r, k] = bf16((q[r, k] - z[r, g]) * scale[r, g]), fp64 [out, in].

    [AWQ-devto, "What do you actually deploy": 4-bit weights used with 16-bit
    activations.] The product (q - z) * scale is exact in fp64 (and in fp32
    while |q - z| < 2^13); bf16 rounding is the only approximation.
    """
    K = np.asarray(qweight).shape[1] * 8
    q = unpack_words(qweight, K).astype(np.float64)
    sc = np.asarray(scales_f16, dtype=np.float16).astype(np.float64)
    z = np.asarray(zeros_f16, dtype=np.float16).astype(np.float64)
    return bf16(dequantize_groups(q, sc, z, group))
