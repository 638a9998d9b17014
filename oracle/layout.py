"""Chunk assignment of the sequence to virtual ranks (oracle side; test infrastructure).

Contiguous: the sequence is cut into c chunks and rank i holds chunk i
("Interrogating parallelism, part 5", section "What breaks the load balance?";
"Context & Expert Parallelism", section "Context parallelism: splitting the
sequence": each device owns a contiguous chunk of tokens).

Zigzag: the sequence is cut into 2c chunks and rank i holds chunks i and
2c-1-i (same section of part 5).  The pages do not say which of a rank's two
chunks comes first in its local memory; the reading taken here is chunk i
first, then chunk 2c-1-i (ascending positions).

"Rank-major" order concatenates the ranks' local rows, rank 0 first.
"""
from __future__ import annotations

import numpy as np


def n_chunks(c: int, layout: int) -> int:
    return c * 2 if layout == 1 else c


def rank_chunks(c: int, layout: int, r: int) -> list[int]:
    """Natural chunk indices held by rank r, in local order."""
    if layout == 1:
        return [r, 2 * c - 1 - r]
    return [r]


def rank_positions(S: int, c: int, layout: int, r: int) -> np.ndarray:
    """Natural sequence positions of rank r's rows, in local order."""
    m = S // n_chunks(c, layout)
    return np.concatenate([np.arange(ch * m, (ch + 1) * m) for ch in rank_chunks(c, layout, r)])


def rank_major_order(S: int, c: int, layout: int) -> np.ndarray:
    """perm[i] = natural position stored at rank-major row i."""
    return np.concatenate([rank_positions(S, c, layout, r) for r in range(c)])


def to_rank_major(x: np.ndarray, S: int, c: int, layout: int) -> np.ndarray:
    """[H, S, ...] natural -> [H, S, ...] rank-major."""
    return x[:, rank_major_order(S, c, layout)]


def from_rank_major(y: np.ndarray, S: int, c: int, layout: int) -> np.ndarray:
    """Inverse of :func:`to_rank_major`."""
    out = np.empty_like(y)
    out[:, rank_major_order(S, c, layout)] = y
    return out
