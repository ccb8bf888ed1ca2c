"""Seeded synthetic linear layers for the AWQ per-layer search.

This module only draws random numbers and rounds them to the storage dtype of
each layer. It holds none of the quantisation method's arithmetic, so both the
CPU oracle (``oracle/``) and the CUDA path can take their inputs from it.

The calibration text and the trained models that the AWQ pages quantise are
not available here, so each layer is synthetic, shaped like the Llama-class
projections the pages have in mind:

* weights ``W[out, in]`` are zero-mean normal with the stated std;
* activations ``X[n_tok, in]`` are a standard normal (or raw Student-t, nu=4)
  bulk in which a fixed set of input channels is multiplied, over every token,
  by one per-channel factor. Outlier channels that persist over nearly every
  token are what "AWQ: How Activation-Aware Quantization Saves 4-bit LLMs"
  describes in "Why does naive 4-bit quantization wreck LLM accuracy?".

Recipe (numpy ``default_rng(seed)``, PCG64), in this order:
  1. ``W = standard_normal((out, in), float32) * w_std``
  2. ``X = standard_normal((n, in), float32)`` (or ``standard_t(4)`` cast to
     float32 for the heavy-tailed bulk)
  3. ``ch = choice(in, k, replace=False)`` with ``k = round(frac * in)``
  4. ``f = uniform(lo, hi, k)`` (or the constant factor), ``X[:, ch] *= f``
  5. ``X`` is rounded to bfloat16 (round-to-nearest-even); ``W`` too when the
     layer stores bf16 weights.
Values are returned as float32 arrays whose entries are exactly the stored
values, plus the bf16 bit patterns where the layer is bf16.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

__all__ = [
    "LayerSpec",
    "LAYERS",
    "WORKLOADS",
    "make_layer",
    "round_to_bf16",
    "bf16_bits",
]


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    """Shape and distribution of one synthetic linear layer."""

    name: str
    out_features: int
    in_features: int
    n_tok: int
    w_std: float
    w_dtype: str  # "fp32" or "bf16"
    x_bulk: str  # "normal" or "t4"
    outlier_count: int
    outlier_lo: float
    outlier_hi: Optional[float]  # None: constant factor outlier_lo
    seed: int

    @property
    def weights(self) -> int:
        return self.out_features * self.in_features


def _k(frac: float, in_features: int) -> int:
    return int(round(frac * in_features))


# The five workloads: tiny; Llama-7B q_proj; Llama-7B MLP pair (up, down);
# 13B-class up_proj; 70B-class MLP.
LAYERS: Dict[str, LayerSpec] = {
    "tiny": LayerSpec("tiny", 256, 256, 128, 0.02, "fp32", "normal", 3, 30.0, None, 0),
    "llama7b_q_proj": LayerSpec(
        "llama7b_q_proj", 4096, 4096, 4096, 0.02, "bf16", "normal", _k(0.01, 4096), 20.0, 50.0, 0
    ),
    "llama7b_mlp_up": LayerSpec(
        "llama7b_mlp_up", 11008, 4096, 4096, 0.02, "bf16", "normal", _k(0.01, 4096), 20.0, 50.0, 0
    ),
    "llama7b_mlp_down": LayerSpec(
        "llama7b_mlp_down", 4096, 11008, 4096, 0.02, "bf16", "normal", _k(0.01, 11008), 20.0, 50.0, 1
    ),
    "13b_up_proj": LayerSpec(
        "13b_up_proj", 13824, 5120, 16384, 0.015, "bf16", "t4", _k(0.01, 5120), 20.0, 80.0, 0
    ),
    "70b_mlp": LayerSpec(
        "70b_mlp", 28672, 8192, 16384, 0.01, "bf16", "t4", _k(0.005, 8192), 50.0, 100.0, 0
    ),
}

# Workload name -> layers it consists of (the MLP pair is two layers).
WORKLOADS: Dict[str, List[str]] = {
    "tiny": ["tiny"],
    "llama7b_q_proj": ["llama7b_q_proj"],
    "llama7b_mlp": ["llama7b_mlp_up", "llama7b_mlp_down"],
    "13b_up_proj": ["13b_up_proj"],
    "70b_mlp": ["70b_mlp"],
}


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); float32 out.

    Inputs are finite, so no NaN handling is needed.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)).astype(np.uint32)
    return r.view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are exactly bf16 (uint16 out)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    if np.any(u & np.uint32(0xFFFF)):
        raise ValueError("values are not exactly representable in bfloat16")
    return (u >> np.uint32(16)).astype(np.uint16)


def make_layer(
    spec: LayerSpec | str,
    *,
    n_tok: Optional[int] = None,
    out_features: Optional[int] = None,
    in_features: Optional[int] = None,
    seed: Optional[int] = None,
) -> Dict[str, object]:
    """Draw one layer. Optional overrides shrink it for small test cases.

    Returns a dict with ``W`` (float32 [out, in]), ``X`` (float32 [n, in],
    bf16-exact), ``w_dtype``, ``outlier_channels`` and ``outlier_factors``.
    """
    if isinstance(spec, str):
        spec = LAYERS[spec]
    out_f = spec.out_features if out_features is None else out_features
    in_f = spec.in_features if in_features is None else in_features
    n = spec.n_tok if n_tok is None else n_tok
    sd = spec.seed if seed is None else seed
    k = spec.outlier_count if in_features is None else max(1, int(round(spec.outlier_count * in_f / spec.in_features)))

    rng = np.random.default_rng(sd)
    W = rng.standard_normal((out_f, in_f), dtype=np.float32)
    W *= np.float32(spec.w_std)
    if spec.x_bulk == "normal":
        X = rng.standard_normal((n, in_f), dtype=np.float32)
    elif spec.x_bulk == "t4":
        X = rng.standard_t(4.0, size=(n, in_f)).astype(np.float32)
    else:
        raise ValueError(spec.x_bulk)
    ch = np.sort(rng.choice(in_f, size=k, replace=False))
    if spec.outlier_hi is None:
        f = np.full(k, spec.outlier_lo, dtype=np.float32)
    else:
        f = rng.uniform(spec.outlier_lo, spec.outlier_hi, size=k).astype(np.float32)
    X[:, ch] *= f[None, :]
    X = round_to_bf16(X)
    if spec.w_dtype == "bf16":
        W = round_to_bf16(W)
    return {
        "name": spec.name,
        "W": W,
        "X": X,
        "w_dtype": spec.w_dtype,
        "outlier_channels": ch,
        "outlier_factors": f,
    }

