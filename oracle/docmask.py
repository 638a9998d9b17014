"""Attention under a document mask over all-gathered keys and values, float64
(oracle side; test infrastructure only).

"Interrogating parallelism, part 5", section "Why did Llama 3 not use a ring?":
Llama 3's context parallelism first all-gathers the key and value tensors and
then computes attention for each rank's local query chunks, because that
composes with any mask -- in particular the document mask, which keeps a token
of a packed sequence from attending across a document boundary.  The query
chunks are the zigzag chunks of "What breaks the load balance?".  Gathering
only moves data, so what every rank computes for its rows is the plain masked
attention below, whatever c and the chunking.

For query head h and natural position i, with doc[i] the document of token i:

    A(i) = { j : j <= i and doc[j] == doc[i] }      (causal inside a document)
    s_j  = sum_t q[h,i,t] * k[h//g, j, t]            j in A(i)
    M    = max_j s_j,   L = sum_j exp(s_j - M)
    out  = sum_j exp(s_j - M) v[h//g, j, :] / L,     lse = M + ln L

Every A(i) holds i itself, so no row is empty.  No 1/sqrt(d) scale, kv head
h // g, as for the ring.
"""
from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):                      # torch tensor (bf16 has no numpy dtype)
        import torch
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def _ids(doc) -> np.ndarray:
    if hasattr(doc, "detach"):
        doc = doc.detach().cpu().numpy()
    return np.asarray(doc).astype(np.int64)


def _rows(qh, kh, vh, doc, pos):
    """Rows ``pos`` of one head: the keys of A(i) lie in [0, max(pos)]."""
    n = int(pos.max()) + 1
    s = qh[pos] @ kh[:n].T                                   # [rows, keys]
    j = np.arange(n)[None, :]
    visible = (j <= pos[:, None]) & (doc[None, :n] == doc[pos][:, None])
    s = np.where(visible, s, -np.inf)
    M = s.max(axis=1)
    e = np.exp(s - M[:, None])
    L = e.sum(axis=1)
    return (e @ vh[:n]) / L[:, None], M + np.log(L)


def doc_attention(q, k, v, doc):
    """q [Hq,S,d], k/v [Hkv,S,d], doc [S] -> out [Hq,S,d], lse [Hq,S] in float64."""
    q, k, v, doc = _f64(q), _f64(k), _f64(v), _ids(doc)
    Hq, S, d = q.shape
    g = Hq // k.shape[0]
    out = np.empty((Hq, S, d))
    lse = np.empty((Hq, S))
    pos = np.arange(S)
    for h in range(Hq):
        out[h], lse[h] = _rows(q[h], k[h // g], v[h // g], doc, pos)
    return out, lse


def doc_attention_rows(q, k, v, doc, heads, positions, batch_rows: int = 256):
    """Selected (head, natural position) rows only, for long sequences."""
    heads = np.asarray(heads, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    doc = _ids(doc)
    g = q.shape[0] // k.shape[0]
    out = np.empty((len(heads), q.shape[2]))
    lse = np.empty(len(heads))
    for h in np.unique(heads):
        idx = np.nonzero(heads == h)[0]
        qh, kh, vh = _f64(q[int(h)]), _f64(k[int(h) // g]), _f64(v[int(h) // g])
        for b0 in range(0, len(idx), batch_rows):
            sel = idx[b0:b0 + batch_rows]
            out[sel], lse[sel] = _rows(qh, kh, vh, doc, positions[sel])
    return out, lse


def doc_pairs(doc) -> int:
    """Visible (query, key) pairs per head: the size of every A(i) added up."""
    doc = _ids(doc)
    total = 0
    for i in range(len(doc)):
        total += int(np.count_nonzero(doc[:i + 1] == doc[i]))
    return total
