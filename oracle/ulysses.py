"""Ulysses sequence parallelism simulated rank by rank, float64 (oracle side; test
infrastructure only).

"Ring Attention and Ulysses shard a sequence two different ways...", section
"Ulysses: an all-to-all relayout instead of a rotation": instead of rotating
key/value blocks past fixed queries, an all-to-all turns the sequence-sharded
layout (each rank: its own tokens, every head) into a head-sharded one (each
rank: a subset of the heads, the whole sequence); attention then runs locally
and completely on each rank's heads, and a second all-to-all turns the result
back.  "Tensor, sequence, context and expert parallelism" (context parallelism
paragraph) says the same: switch from splitting by sequence to splitting by
heads for attention, then switch back.

Readings (the pages fix none of these):
* a rank's sequence shard is its ring chunk(s), contiguous or zigzag, in the
  local order of :mod:`oracle.layout` (chunk i, then chunk 2c-1-i);
* a sequence-sharded tensor is token-major, [tokens, H, row] on each rank (the
  layout of an activation), and the ranks' shards concatenated rank 0 first give
  [S, H, row] in rank-major token order;
* after the all-to-all, rank r holds the query heads [r*Hq/c, (r+1)*Hq/c) in
  head-major natural order [heads, S, row], so Hq % c == 0; for keys and values
  it holds the KV heads its query heads use (h // g), which replicates a KV head
  on c/Hkv ranks when c > Hkv;
* the attention on each rank is the full-sequence attention of
  :mod:`oracle.attention` on its heads (no 1/sqrt(d), kv head h // g).
"""
from __future__ import annotations

import numpy as np

from oracle import attention, layout


def q_heads(Hq: int, c: int, r: int) -> np.ndarray:
    """Query heads held by rank r after the relayout."""
    per = Hq // c
    return np.arange(r * per, (r + 1) * per)


def kv_heads(Hq: int, Hkv: int, c: int, r: int) -> np.ndarray:
    """KV heads rank r needs: those of its query heads."""
    g = Hq // Hkv
    return np.unique(q_heads(Hq, c, r) // g)


def seq_to_heads(shards: list, heads_of, S: int, c: int, lay: int) -> list:
    """All-to-all, sequence-sharded -> head-sharded, message by message.

    ``shards[r]``: rank r's [n_r, H, row] tokens in local order.  ``heads_of(r)``:
    the heads receiver r keeps.  Sender s sends receiver r the columns heads_of(r)
    of its tokens; r writes each received token at its natural position.  Returns
    one [len(heads_of(r)), S, row] array per rank.
    """
    row = shards[0].shape[2:]
    out = [np.zeros((len(heads_of(r)), S) + row) for r in range(c)]
    for s in range(c):
        pos = layout.rank_positions(S, c, lay, s)        # natural position of each local token
        for r in range(c):
            msg = shards[s][:, heads_of(r)]                # [n_s, heads of r, row]
            out[r][:, pos] = np.swapaxes(msg, 0, 1)
    return out


def heads_to_seq(parts: list, heads_of, H: int, S: int, c: int, lay: int) -> list:
    """The inverse all-to-all: ``parts[r]`` is rank r's [heads_of(r), S, row] result;
    returns each rank's [n_r, H, row] sequence shard with every head."""
    row = parts[0].shape[2:]
    shards = []
    for s in range(c):
        pos = layout.rank_positions(S, c, lay, s)
        x = np.zeros((len(pos), H) + row)
        for r in range(c):
            x[:, heads_of(r)] = np.swapaxes(parts[r][:, pos], 0, 1)
        shards.append(x)
    return shards


def split_shards(x_seq: np.ndarray, c: int) -> list:
    """[S, H, row] rank-major token order -> list of c rank shards."""
    n_r = x_seq.shape[0] // c
    return [x_seq[r * n_r:(r + 1) * n_r] for r in range(c)]


def ulysses_attention(q_seq, k_seq, v_seq, c: int, lay: int, causal: bool):
    """Sequence-sharded q [S, Hq, d], k, v [S, Hkv, d] (rank-major token order) ->
    sequence-sharded out [S, Hq, d] and lse [S, Hq]: relayout, full-sequence
    attention per rank on its heads, relayout back."""
    q_seq, k_seq, v_seq = (np.asarray(x, dtype=np.float64) for x in (q_seq, k_seq, v_seq))
    S, Hq, _ = q_seq.shape
    Hkv = k_seq.shape[1]
    g = Hq // Hkv
    qh = seq_to_heads(split_shards(q_seq, c), lambda r: q_heads(Hq, c, r), S, c, lay)
    kh = seq_to_heads(split_shards(k_seq, c), lambda r: kv_heads(Hq, Hkv, c, r), S, c, lay)
    vh = seq_to_heads(split_shards(v_seq, c), lambda r: kv_heads(Hq, Hkv, c, r), S, c, lay)
    outs, lses = [], []
    for r in range(c):
        # each query head's KV head, as an index into this rank's KV heads
        local_kv = np.searchsorted(kv_heads(Hq, Hkv, c, r), q_heads(Hq, c, r) // g)
        o = np.empty(qh[r].shape)
        l = np.empty(qh[r].shape[:2])
        for i, j in enumerate(local_kv):
            oi, li = attention.full_attention(qh[r][i:i + 1], kh[r][j:j + 1], vh[r][j:j + 1], causal)
            o[i], l[i] = oi[0], li[0]
        outs.append(o)
        lses.append(l[..., None])
    out = heads_to_seq(outs, lambda r: q_heads(Hq, c, r), Hq, S, c, lay)
    lse = heads_to_seq(lses, lambda r: q_heads(Hq, c, r), Hq, S, c, lay)
    return np.concatenate(out), np.concatenate(lse)[..., 0]
