"""Per-rank causal work (oracle side; test infrastructure).

"Interrogating parallelism, part 5" (section "What breaks the load balance?")
counts work in chunk units: with c contiguous chunks rank i does i+1 units,
so the last rank does c times the first; with 2c zigzag chunks rank i does
(i+1) + (2c-i) = 2c+1 units, the same for every rank.  A unit there is one
(query chunk, key chunk) pair with any visible key, the diagonal pair counted
whole.

Three counts per rank, each computed from its definition by enumeration:

* ``units`` -- (query chunk, key chunk) pairs with at least one visible
  (query, key) pair; chunks are the layout's chunks (c or 2c of them).
* ``pairs`` -- visible (query, key) pairs: sum over the rank's queries of the
  number of keys it attends to.
* ``tiles`` -- (query tile, key tile) pairs with at least one visible pair,
  tiles being ``tile`` consecutive rows of the rank's local query rows and of
  each chunk of keys.
"""
from __future__ import annotations

import numpy as np

from .layout import n_chunks, rank_chunks, rank_positions


def rank_work(S: int, c: int, causal: bool, layout: int, tile: int = 128):
    nch = n_chunks(c, layout)
    m = S // nch
    units, pairs, tiles = [], [], []
    for r in range(c):
        mine = rank_chunks(c, layout, r)
        u = 0
        for qc in mine:
            for kc in range(nch):
                # chunk kc has a key visible to chunk qc iff its first key <= qc's last query
                if not causal or kc * m <= qc * m + m - 1:
                    u += 1
        units.append(u)
        pos = rank_positions(S, c, layout, r)
        pairs.append(int(np.sum(pos + 1)) if causal else len(pos) * S)
        t = 0
        for t0 in range(0, len(pos), tile):
            qmax = pos[t0:t0 + tile].max()
            for kc in range(nch):
                for k0 in range(kc * m, kc * m + m, tile):
                    if not causal or k0 <= qmax:
                        t += 1
        tiles.append(t)
    return np.array(units), np.array(pairs, dtype=np.int64), np.array(tiles, dtype=np.int64)
