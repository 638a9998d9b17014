"""Helpers for the GPU parity tests: device tensors from the seeded generators,
oracle comparisons, tolerances."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances (max abs error over all checked elements):
#   fp32 path: 1e-5 on out and lse;
#   bf16 path: 2e-2 on out, 1e-3 on lse;
#   permutation: bit-exact.
TOL_F32 = 1e-5
TOL_BF16_OUT = 2e-2
TOL_BF16_LSE = 1e-3


def dev():
    return torch.device("cuda:0")


def rank_major(x: torch.Tensor, S: int, c: int, layout: int) -> torch.Tensor:
    """Natural -> rank-major on the host by plain indexing (test side, no library call)."""
    from oracle.layout import rank_major_order
    idx = torch.from_numpy(rank_major_order(S, c, layout))
    return x[:, idx].contiguous()


def natural(y: torch.Tensor, S: int, c: int, layout: int) -> torch.Tensor:
    from oracle.layout import rank_major_order
    idx = torch.from_numpy(rank_major_order(S, c, layout))
    out = torch.empty_like(y)
    out[:, idx] = y
    return out


def max_err(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_ninf = np.isneginf(a) & np.isneginf(b)
    with np.errstate(invalid="ignore"):
        d = np.where(both_ninf, 0.0, np.abs(a - b))
    return float(np.nan_to_num(d, nan=np.inf).max()) if d.size else 0.0


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()
