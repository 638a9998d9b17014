"""Full-row softmax attention in float64 (oracle side; test infrastructure).

This is the plain definition that ring attention reaches exactly: the ring's
merged partial results are identical to ordinary softmax attention over the
whole row ("Interrogating parallelism, part 5", section "How does attention
survive being split?"; the worked example in "Ring Attention and Ulysses
shard a sequence two different ways..." computes this reference with
``q @ k_full.T``, a row max, exponentials and a row sum).

For query head h, natural position i and key set A(i):

    s_j   = sum_t q[h,i,t] * k[h//g, j, t]        j in A(i)
    M     = max_j s_j
    L     = sum_j exp(s_j - M)
    out   = sum_j exp(s_j - M) * v[h//g, j, :] / L
    lse   = M + ln L

A(i) = {j <= i} when causal ("Context & Expert Parallelism": token i must
attend to every token j <= i), else all j.  No 1/sqrt(d) scale is applied:
the pages' update rule uses ``scores = q @ k.T`` as is.  Grouped-query heads
map consecutively, kv head = h // g with g = Hq / Hkv (the pages give only
the head counts, 64 query heads against 8 KV heads).
"""
from __future__ import annotations

import numpy as np


def _head_rows(qh: np.ndarray, kh: np.ndarray, vh: np.ndarray, pos: np.ndarray, causal: bool):
    """Rows ``pos`` of one head; keys 0..max(pos) suffice when causal."""
    n_keys = int(pos.max()) + 1 if causal else kh.shape[0]
    s = qh[pos] @ kh[:n_keys].T                           # [rows, keys]
    if causal:
        s = np.where(np.arange(n_keys)[None, :] > pos[:, None], -np.inf, s)
    M = s.max(axis=1)
    e = np.exp(s - M[:, None])
    L = e.sum(axis=1)
    out = (e @ vh[:n_keys]) / L[:, None]
    lse = M + np.log(L)
    return out, lse


def full_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool):
    """q [Hq,S,d], k/v [Hkv,S,d] (any float dtype) -> out [Hq,S,d], lse [Hq,S] in float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Hq, S, d = q.shape
    g = Hq // k.shape[0]
    out = np.empty((Hq, S, d))
    lse = np.empty((Hq, S))
    pos = np.arange(S)
    for h in range(Hq):
        out[h], lse[h] = _head_rows(q[h], k[h // g], v[h // g], pos, causal)
    return out, lse


def full_attention_rows(q, k, v, heads, positions, causal: bool, batch_rows: int = 256):
    """Selected (head, natural position) rows only, for sequences too long to do whole.

    ``q``/``k``/``v`` may be torch or numpy arrays of any float dtype; they are
    upcast exactly to float64 one head at a time.
    """
    heads = np.asarray(heads, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    Hq = q.shape[0]
    g = Hq // k.shape[0]
    d = q.shape[2]
    out = np.empty((len(heads), d))
    lse = np.empty(len(heads))
    for h in np.unique(heads):
        idx = np.nonzero(heads == h)[0]
        qh = _as_f64(q[int(h)])
        kh = _as_f64(k[int(h) // g])
        vh = _as_f64(v[int(h) // g])
        for b0 in range(0, len(idx), batch_rows):
            sel = idx[b0:b0 + batch_rows]
            out[sel], lse[sel] = _head_rows(qh, kh, vh, positions[sel], causal)
    return out, lse


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):                      # torch tensor (bf16 has no numpy dtype)
        import torch
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)
