"""Seeded synthetic inputs for the ring-attention hot path.

This module draws random tensors and nothing else: it holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it without sharing any of the method.

The worked example in "Ring Attention and Ulysses shard a sequence two
different ways..." (section "Ring Attention: point-to-point rotation, and an
online softmax that never sees the whole row at once") draws q, K and V from
N(0, 1) without a seed; here every draw comes from a torch CPU generator with
a fixed seed so that results repeat:

    Q: seed 0, K: seed 1, V: seed 2, Q outlier mask: seed 3, K outlier mask:
    seed 4, document lengths: seed 5, sampled query rows: seed 1234.

Tensors are head-major and in natural sequence order, ``[B*H, S, d]``.
"""
from __future__ import annotations

import torch

SEED_Q, SEED_K, SEED_V = 0, 1, 2
SEED_Q_MASK, SEED_K_MASK = 3, 4
SEED_DOCS = 5
SEED_ROWS = 1234


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def normal(shape, seed: int) -> torch.Tensor:
    """N(0, 1) float32 on the CPU from a fresh generator seeded with ``seed``."""
    return torch.randn(shape, generator=_gen(seed), dtype=torch.float32)


def outlier_scale(x: torch.Tensor, seed: int, frac: float, factor: float) -> torch.Tensor:
    """Multiply an i.i.d. Bernoulli(``frac``) subset of entries by ``factor``.

    The mask is drawn from its own generator (``seed``) so that Q and K get
    independent masks.
    """
    u = torch.rand(x.shape, generator=_gen(seed), dtype=torch.float32)
    return torch.where(u < frac, x * factor, x)


def make_qkv(w) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Q, K, V on the CPU for workload ``w`` (a :class:`configs.Workload`).

    Steps: N(0,1) float32 -> optional outlier scaling of Q and K -> optional
    scale of Q in float32 -> cast to the workload's dtype.  The same cast
    bytes feed the device and the oracle.
    """
    bhq, bhkv = w.batch * w.hq, w.batch * w.hkv
    q = normal((bhq, w.seq, w.d), SEED_Q)
    k = normal((bhkv, w.seq, w.d), SEED_K)
    v = normal((bhkv, w.seq, w.d), SEED_V)
    if w.outlier_frac > 0.0:
        q = outlier_scale(q, SEED_Q_MASK, w.outlier_frac, w.outlier_factor)
        k = outlier_scale(k, SEED_K_MASK, w.outlier_frac, w.outlier_factor)
    if w.q_scale != 1.0:
        q = q * w.q_scale
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    return q.to(dt).contiguous(), k.to(dt).contiguous(), v.to(dt).contiguous()


def doc_ids(seq: int, lo: int, hi: int, seed: int = SEED_DOCS) -> torch.Tensor:
    """Document id of every position of a packed sequence, int32 [seq], non-decreasing.

    Documents are laid end to end; their lengths are drawn log-uniformly from
    [lo, hi] (many short documents, a few long ones) until ``seq`` tokens are
    filled, and the last one is cut to fit.  Ids count 0, 1, 2, ... in order.
    """
    g = _gen(seed)
    ids = torch.empty(seq, dtype=torch.int32)
    pos, doc = 0, 0
    llo, lhi = float(torch.log(torch.tensor(float(lo)))), float(torch.log(torch.tensor(float(hi) + 1.0)))
    while pos < seq:
        u = float(torch.rand((), generator=g))
        n = int(torch.exp(torch.tensor(llo + u * (lhi - llo))))
        n = max(lo, min(hi, n, seq - pos))
        ids[pos:pos + n] = doc
        pos += n
        doc += 1
    return ids


def sample_rows(bh: int, seq: int, n: int, seed: int = SEED_ROWS) -> tuple[torch.Tensor, torch.Tensor]:
    """``n`` distinct (head, position) pairs, uniform without replacement."""
    total = bh * seq
    n = min(n, total)
    flat = torch.randperm(total, generator=_gen(seed))[:n]
    flat, _ = torch.sort(flat)
    return (flat // seq).to(torch.int64), (flat % seq).to(torch.int64)


def edge_rows(bh: int, seq: int, n_chunks: int) -> tuple[torch.Tensor, torch.Tensor]:
    """Rows where indexing mistakes show first: positions 0 and S-1 and the
    first and last row of every natural chunk, for heads 0 and bh-1."""
    m = seq // n_chunks
    pos = {0, seq - 1}
    for ch in range(n_chunks):
        pos.add(ch * m)
        pos.add(ch * m + m - 1)
    heads = sorted({0, bh - 1})
    hs, ps = [], []
    for h in heads:
        for p in sorted(pos):
            hs.append(h)
            ps.append(p)
    return torch.tensor(hs, dtype=torch.int64), torch.tensor(ps, dtype=torch.int64)
