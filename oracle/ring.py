"""The per-rank ring computation, restated step by step in float64 (oracle side).

Follows "Ring Attention and Ulysses shard a sequence two different ways..."
(section "Ring Attention: point-to-point rotation, and an online softmax that
never sees the whole row at once"): each rank keeps its queries fixed and
works through the KV blocks as they arrive, one online update per block:

    block_max   = row max of the block's scores
    new_max     = max(running_max, block_max)
    correction  = exp(running_max - new_max)
    p           = exp(scores - new_max)
    running_sum = running_sum * correction + row sum of p
    output      = output * correction + p @ V_block
    running_max = new_max

and divides by the running sum at the end.  The ring order is taken from
"Interrogating parallelism, part 5" (section "How does attention survive being
split?"): rank i sends its KV block to rank i+1, so at hop h rank r holds the
block that rank (r - h) mod c started with; after c-1 hops every query block
has seen every KV block.

Readings where the pages are silent:

* A rank's KV block is its own chunk (contiguous) or its two chunks (zigzag).
  A "ring message" of ``kv_block`` rows is the unit of one online update; the
  block must divide a chunk.
* Causal masking uses natural positions (key j is visible to query i when
  j <= i).  A row whose keys in a block are all masked takes no update from
  that block (the printed rule would form exp(-inf - (-inf)) there).
* The log-sum-exp of a row is running_max + ln(running_sum); a row that saw no
  key at all has output 0 and log-sum-exp -inf.
"""
from __future__ import annotations

import numpy as np

from .layout import rank_positions


def ring_rank(q_rows, q_pos, k, v, kv_blocks_pos, causal: bool):
    """One rank: queries ``q_rows`` at natural positions ``q_pos`` visit the
    key/value rows at the natural positions listed in ``kv_blocks_pos``, one
    online update per list entry, in list order."""
    n, _ = q_rows.shape
    dv = v.shape[1]
    running_max = np.full(n, -np.inf)
    running_sum = np.zeros(n)
    output = np.zeros((n, dv))
    with np.errstate(invalid="ignore", over="ignore"):
        for pos_k in kv_blocks_pos:
            scores = q_rows @ k[pos_k].T
            if causal:
                scores = np.where(pos_k[None, :] > q_pos[:, None], -np.inf, scores)
            block_max = scores.max(axis=1)
            new_max = np.maximum(running_max, block_max)
            seen = np.isfinite(new_max)          # rows with at least one visible key so far
            correction = np.where(seen, np.exp(running_max - new_max), 1.0)
            p = np.where(seen[:, None], np.exp(scores - new_max[:, None]), 0.0)
            running_sum = running_sum * correction + p.sum(axis=1)
            output = output * correction[:, None] + p @ v[pos_k]
            running_max = new_max
    seen = running_sum > 0
    out = np.where(seen[:, None], output / np.where(seen, running_sum, 1.0)[:, None], 0.0)
    with np.errstate(divide="ignore"):
        lse = np.where(seen, running_max + np.log(np.where(seen, running_sum, 1.0)), -np.inf)
    return out, lse


def ring_schedule(S: int, c: int, layout: int, r: int, kv_block: int, hops=None):
    """Natural key positions of every ring message rank r receives, in order.

    ``hops`` restricts the schedule to the listed hop indices (all c by default).
    """
    msgs = []
    for h in (range(c) if hops is None else hops):
        src = (r - h) % c
        block = rank_positions(S, c, layout, src)
        for s0 in range(0, len(block), kv_block):
            msgs.append(block[s0:s0 + kv_block])
    return msgs


def ring_attention(q, k, v, c: int, layout: int, causal: bool, kv_block: int):
    """All c ranks; returns out [Hq,S,d] and lse [Hq,S] in natural order, float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Hq, S, d = q.shape
    g = Hq // k.shape[0]
    out = np.zeros((Hq, S, v.shape[2]))
    lse = np.zeros((Hq, S))
    for h in range(Hq):
        for r in range(c):
            pos = rank_positions(S, c, layout, r)
            o, l = ring_rank(q[h, pos], pos, k[h // g], v[h // g],
                             ring_schedule(S, c, layout, r, kv_block), causal)
            out[h, pos] = o
            lse[h, pos] = l
    return out, lse


def ring_hop_partial(q, k, v, c: int, layout: int, causal: bool, kv_block: int, hop: int, sub: int):
    """The partial each rank forms from one ring message: hop ``hop``,
    sub-block ``sub`` of the KV block held at that hop.  Returns
    (out, lse) in natural order; rows with no visible key get 0 and -inf."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Hq, S, d = q.shape
    g = Hq // k.shape[0]
    out = np.zeros((Hq, S, v.shape[2]))
    lse = np.zeros((Hq, S))
    for h in range(Hq):
        for r in range(c):
            pos = rank_positions(S, c, layout, r)
            msg = ring_schedule(S, c, layout, r, kv_block, hops=[hop])[sub]
            o, l = ring_rank(q[h, pos], pos, k[h // g], v[h // g], [msg], causal)
            out[h, pos] = o
            lse[h, pos] = l
    return out, lse
