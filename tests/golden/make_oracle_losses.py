"""Write the oracle's per-alpha losses for the full-size workloads.

Calls only ``oracle`` and the seeded generator ``workloads``; nothing here
touches the CUDA path. The loss of a layer is a sum over its output rows, so
the rows are taken in blocks (each block is the oracle's plain definition on a
sub-layer) and the block sums are added in order before dividing by
n_tok * out_features.

Usage:  python tests/golden/make_oracle_losses.py [layer ...]
Output: tests/golden/oracle_losses.json (merged with what is already there).
"""
import hashlib
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle as O  # noqa: E402
import workloads  # noqa: E402

OUT = os.path.join(HERE, "oracle_losses.json")
N_GRID = 20
ROW_BLOCK = 2048


def digest(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()[:16]


def layer_losses(name: str) -> dict:
    L = workloads.make_layer(name)
    W32, X32 = L["W"], L["X"]
    X = X32.astype(np.float64)
    n, N = X.shape[0], W32.shape[0]
    sx = O.channel_importance(X)
    losses = []
    for i, alpha in enumerate(O.alpha_grid(N_GRID)):
        s = O.awq_scales(sx, alpha)
        total = 0.0
        for r0 in range(0, N, ROW_BLOCK):
            Wb = W32[r0:r0 + ROW_BLOCK].astype(np.float64)
            total += O.output_sq_err_sum(X, Wb, O.fake_quantize(Wb, s))
        losses.append(total / (n * N))
        print(f"{name} alpha[{i}]={alpha:.2f} loss={losses[-1]:.9e}", flush=True)
    best_i, best = -1, float("inf")
    for i, v in enumerate(losses):
        if v < best:
            best_i, best = i, v
    return {
        "n_tok": n,
        "out_features": N,
        "in_features": X.shape[1],
        "n_grid": N_GRID,
        "losses": losses,
        "best_idx": best_i,
        "W_sha256_16": digest(W32),
        "X_sha256_16": digest(X32),
    }


def main(names):
    data = {}
    if os.path.exists(OUT):
        data = json.load(open(OUT))
    data.setdefault("_source", "oracle/awq_oracle.py via tests/golden/make_oracle_losses.py; "
                    "inputs from workloads.make_layer (seeded)")
    for name in names:
        t = time.time()
        data[name] = layer_losses(name)
        data[name]["oracle_seconds"] = round(time.time() - t, 1)
        with open(OUT, "w") as f:
            json.dump(data, f, indent=1, sort_keys=True)
        print(f"{name}: done in {time.time() - t:.0f}s", flush=True)


if __name__ == "__main__":
    names = sys.argv[1:] or [k for k in workloads.LAYERS if k != "tiny"]
    main(names)
