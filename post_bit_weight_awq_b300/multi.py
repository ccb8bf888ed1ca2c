"""Host-side logic for running the AWQ search on several GPUs of one node.

Two ways to use N GPUs, both one process per GPU:

* independent layers (what the benchmark does): every rank quantises its own
  layer; no data crosses between ranks, and only the timing is reduced
  (``max_over_ranks``);
* one layer split by output rows: s depends only on X and the squared error
  is a sum over output rows ("AWQ: How Activation-Aware Quantization Saves
  4-bit LLMs", search_scale listing: the mean over the whole output), so each
  rank searches its block of rows and a single all-reduce of n_grid sums
  gives every rank the whole layer's losses and the same first-minimum alpha
  (``combine_row_shards``). The final pack of each block is then local.

These functions take a ``torch.distributed`` process group and work with
any backend (NCCL on GPUs, gloo on CPU for the tests).
"""
from __future__ import annotations

from typing import Sequence, Tuple

import torch
import torch.distributed as dist


def shard_rows(out_features: int, world: int, rank: int) -> Tuple[int, int]:
    """Contiguous block of output rows [r0, r1) owned by ``rank``; sizes
    differ by at most one row."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    base, extra = divmod(out_features, world)
    r0 = rank * base + min(rank, extra)
    return r0, r0 + base + (1 if rank < extra else 0)


def combine_row_shards(shard_losses: Sequence[float], n_tok: int, shard_rows_count: int, out_features: int,
                       group=None):
    """Whole-layer per-alpha losses from every rank's block losses.

    ``shard_losses[i]`` is the mean squared error of the rank's block for
    alpha_i (mean over n_tok * shard_rows_count). Returns (losses, best_idx)
    identical on every rank: losses[i] = sum over ranks of block sums /
    (n_tok * out_features), best_idx = first strict minimum.
    """
    sums = torch.tensor([float(v) * n_tok * shard_rows_count for v in shard_losses], dtype=torch.float64)
    dist.all_reduce(sums, op=dist.ReduceOp.SUM, group=group)
    losses = (sums / (float(n_tok) * float(out_features))).tolist()
    best, best_v = 0, float("inf")
    for i, v in enumerate(losses):
        if v < best_v:
            best, best_v = i, v
    return losses, best


def max_over_ranks(value: float, group=None, device=None) -> float:
    """Largest ``value`` over the ranks (the job's time is its slowest rank)."""
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())
