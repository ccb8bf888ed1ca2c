"""One-call AWQ quantisation of a linear layer on the GPU.

Allocates the outputs and the scratch with torch (device memory only) and
runs the three library steps on the current stream: activation statistics,
the alpha grid search, and the final INT4 pack. Every computation happens in
libawq.so's kernels.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

from . import capi


@dataclasses.dataclass
class QuantizedLayer:
    mean_abs: torch.Tensor  # fp32 [in]
    losses: torch.Tensor  # fp32 [n_grid]
    best_idx: torch.Tensor  # int32 [1]
    s_best: torch.Tensor  # fp32 [in]; fold 1/s_best into the producer of X
    qweight: torch.Tensor  # int32 [out, in * w_bit / 32]
    scales: torch.Tensor  # fp16 [out, in/group]
    zeros: torch.Tensor  # fp16 [out, in/group]
    row_losses: Optional[torch.Tensor] = None  # fp32 [n_grid, out] when asked for: each row's share of the loss


class Workspace:
    """Device scratch reused across calls (grown on demand)."""

    def __init__(self, device=None):
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self.buf = torch.empty(0, dtype=torch.uint8, device=self.device)

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        return self.buf


def _check_inputs(W: torch.Tensor, X: torch.Tensor) -> None:
    if not (W.is_cuda and X.is_cuda):
        raise ValueError("W and X must be CUDA tensors")
    if not (W.is_contiguous() and X.is_contiguous()):
        raise ValueError("W and X must be contiguous row-major")
    if X.dtype != torch.bfloat16:
        raise ValueError("X must be bfloat16")
    if W.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("W must be bfloat16 or float32")
    if W.shape[1] != X.shape[1]:
        raise ValueError("W and X disagree on in_features")


def quantize_layer(W: torch.Tensor, X: torch.Tensor, cfg: Optional[capi.AwqConfig] = None,
                   workspace: Optional[Workspace] = None, stream=None, row_losses: bool = False) -> QuantizedLayer:
    """AWQ search + INT4 pack of one layer (asynchronous on ``stream``); with ``row_losses`` the search
    also returns each output row's share of every alpha's loss."""
    _check_inputs(W, X)
    cfg = capi.config() if cfg is None else cfg
    N, K = W.shape
    n = X.shape[0]
    dev = W.device
    ws = workspace if workspace is not None else Workspace(dev)
    need = max(capi.awq_workspace_size(n, N, K, cfg), capi.awq_act_stats_workspace_size(n, K))
    buf = ws.get(need)
    out = QuantizedLayer(
        mean_abs=torch.empty(K, dtype=torch.float32, device=dev),
        losses=torch.empty(cfg.n_grid, dtype=torch.float32, device=dev),
        best_idx=torch.empty(1, dtype=torch.int32, device=dev),
        s_best=torch.empty(K, dtype=torch.float32, device=dev),
        qweight=torch.empty(N, K * cfg.w_bit // 32, dtype=torch.int32, device=dev),
        scales=torch.empty(N, K // cfg.group, dtype=torch.float16, device=dev),
        zeros=torch.empty(N, K // cfg.group, dtype=torch.float16, device=dev),
        row_losses=torch.empty(cfg.n_grid, N, dtype=torch.float32, device=dev) if row_losses else None,
    )
    capi.awq_act_stats(X, out.mean_abs, buf, stream)
    capi.awq_search_layer(W, X, out.mean_abs, cfg, out.losses, out.best_idx, out.s_best, buf, stream,
                          row_losses=out.row_losses)
    capi.awq_quantize_pack(W, out.s_best, cfg, out.qweight, out.scales, out.zeros, stream)
    return out
