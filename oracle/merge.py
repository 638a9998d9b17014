"""Exact combination of two attention partials (oracle side; test infrastructure).

"Interrogating parallelism, part 5" (section "How does attention survive
being split?") states that attention over one block of keys, kept with its
running max and sum, combines with attention over another block exactly.
Written with each partial as a normalised output ``o`` and its log-sum-exp
``lse`` (the reading taken here; the pages keep max and sum separately, and
lse = max + ln sum carries the same information):

    lse = ln(exp(lse_a) + exp(lse_b))
    o   = o_a * exp(lse_a - lse) + o_b * exp(lse_b - lse)

A partial with lse = -inf saw no key and has weight 0; if both are -inf the
result is o = 0, lse = -inf.
"""
from __future__ import annotations

import numpy as np


def merge(o_a, lse_a, o_b, lse_b):
    o_a = np.asarray(o_a, dtype=np.float64)
    o_b = np.asarray(o_b, dtype=np.float64)
    lse_a = np.asarray(lse_a, dtype=np.float64)
    lse_b = np.asarray(lse_b, dtype=np.float64)
    M = np.maximum(lse_a, lse_b)
    empty = ~np.isfinite(M)
    Ms = np.where(empty, 0.0, M)
    ea = np.exp(lse_a - Ms)
    eb = np.exp(lse_b - Ms)
    tot = ea + eb
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(empty, -np.inf, Ms + np.log(tot))
        wa = np.where(empty, 0.0, ea / tot)
        wb = np.where(empty, 0.0, eb / tot)
    return o_a * wa[..., None] + o_b * wb[..., None], lse
