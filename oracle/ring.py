"""The per-rank ring computation, restated step by step in float64 (oracle side; test
infrastructure only).

Follows "Ring Attention and Ulysses shard a sequence two different ways..."
(section "Ring Attention: point-to-point rotation, and an online softmax that
never sees the whole row at once"): each rank keeps its queries fixed and
works through the KV blocks as they arrive.  What a rank carries between
blocks, per query row, is a reference maximum ``m``, the sum ``l`` of the
exponentials of the scores seen so far taken against ``m``, and the matching
weighted sum ``acc`` of value rows.  One arriving block is absorbed in the
order the page's update rule gives:

1. the block's largest score per row;
2. the new reference: the larger of that and the old one;
3. the factor that moves everything accumulated so far onto the new
   reference, e raised to (old reference - new reference);
4. the block's exponentials against the new reference;
5. ``l`` and ``acc`` rescaled by that factor, the block's exponentials (and
   their product with the block's values) added;
6. the new reference kept.

At the end out = acc / l and the log-sum-exp is m + ln l.  The ring order is
taken from "Interrogating parallelism, part 5" (section "How does attention
survive being split?"): rank i sends its KV block to rank i+1, so at hop h
rank r holds the block that rank (r - h) mod c started with; after c-1 hops
every query block has seen every KV block.

Readings where the pages are silent:

* A rank's KV block is its own chunk (contiguous) or its two chunks (zigzag).
  A "ring message" of ``kv_block`` rows is the unit of one online update; the
  block must divide a chunk.
* Causal masking uses natural positions (key j is visible to query i when
  j <= i).  A row whose keys in a block are all masked takes no update from
  that block (the printed rule would form exp(-inf - (-inf)) there).
* The log-sum-exp of a row is m + ln(l); a row that saw no key at all has
  output 0 and log-sum-exp -inf.
"""
from __future__ import annotations

import numpy as np

from .layout import rank_positions


class _RowState:
    """Per-row online-softmax state of one rank's queries: reference maximum m,
    exponential sum l and weighted value sum acc, all relative to m."""

    def __init__(self, n_rows: int, d_v: int):
        self.m = np.full(n_rows, -np.inf)
        self.l = np.zeros(n_rows)
        self.acc = np.zeros((n_rows, d_v))

    def absorb(self, scores: np.ndarray, values: np.ndarray) -> None:
        """Fold one block in: ``scores`` [rows, keys] (-inf where masked),
        ``values`` [keys, d_v]."""
        top = scores.max(axis=1)                                 # step 1
        ref = np.maximum(self.m, top)                            # step 2
        live = ref > -np.inf        # rows that have met a visible key by now
        safe_ref = np.where(live, ref, 0.0)
        with np.errstate(invalid="ignore"):
            # step 3; a row that had seen nothing yet has l = acc = 0, and any
            # finite factor leaves that as it is
            alpha = np.where(live & (self.m > -np.inf), np.exp(self.m - safe_ref), 0.0)
        w = np.exp(scores - safe_ref[:, None])                   # step 4 (masked: 0)
        w[~live] = 0.0
        self.l = alpha * self.l + w.sum(axis=1)                  # step 5
        self.acc = alpha[:, None] * self.acc + w @ values
        self.m = ref                                             # step 6

    def finish(self):
        """(out, lse) of every row; out = 0 and lse = -inf for a row that saw no key."""
        have = self.l > 0
        den = np.where(have, self.l, 1.0)
        out = np.where(have[:, None], self.acc / den[:, None], 0.0)
        lse = np.where(have, np.where(have, self.m, 0.0) + np.log(den), -np.inf)
        return out, lse


def ring_rank(q_rows, q_pos, k, v, kv_blocks_pos, causal: bool):
    """One rank: queries ``q_rows`` at natural positions ``q_pos`` visit the
    key/value rows at the natural positions listed in ``kv_blocks_pos``, one
    online update per list entry, in list order."""
    state = _RowState(q_rows.shape[0], v.shape[1])
    for keys in kv_blocks_pos:
        blk = q_rows @ k[keys].T
        if causal:
            blk = np.where(keys[None, :] <= q_pos[:, None], blk, -np.inf)
        state.absorb(blk, v[keys])
    return state.finish()


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
