"""Helpers shared by the GPU tests: device upload of generator output and
diagnostic dumps. No method arithmetic lives here."""
import os

import numpy as np
import torch

import workloads


def dev_bf16(a32: np.ndarray) -> torch.Tensor:
    """Upload float32 values that are exactly bf16 as a bf16 CUDA tensor."""
    bits = workloads.bf16_bits(a32)
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def dev_f32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def dev_weight(L) -> torch.Tensor:
    return dev_bf16(L["W"]) if L["w_dtype"] == "bf16" else dev_f32(L["W"])


def host_bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    """bf16 CUDA tensor -> float64 numpy (exact)."""
    bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def save_debug(name: str, **arrays) -> None:
    """On a failing check, keep the arrays for offline diagnosis in the
    folder named by AWQ_DEBUG_DIR (nothing is written when it is unset)."""
    out = os.environ.get("AWQ_DEBUG_DIR")
    if out and os.path.isdir(out):
        np.savez_compressed(os.path.join(out, f"debug_{name}.npz"), **arrays)
