"""Gradients of the attention the ring computes, float64 (oracle side; test
infrastructure only).

The pages do not describe a backward pass; they count it only through the
training FLOP estimate of "Interrogating parallelism, part 5" (forward plus
backward).  The reading taken here: the backward pass of ring attention is the
exact gradient of the forward of :mod:`oracle.attention` -- out_i = sum_j
softmax_j(q_i . k_j) v_j over the visible keys, no 1/sqrt(d), kv head h // g --
with respect to q, k and v, given the gradient dout of the output.  Writing
P_ij = exp(q_i . k_j - lse_i) for visible pairs (0 otherwise):

    dV_j  = sum_i P_ij dout_i
    dP_ij = dout_i . v_j
    D_i   = sum_j P_ij dP_ij  = dout_i . out_i
    dS_ij = P_ij (dP_ij - D_i)
    dQ_i  = sum_j dS_ij k_j,      dK_j = sum_i dS_ij q_i

and a KV head's dK, dV sum over the query heads that use it.

:func:`ring_backward` restates how a ring computes it: every rank keeps its
queries, dout, lse and D fixed (as in the forward, "How does attention survive
being split?"), and each KV block travels around the ring together with its dK,
dV accumulators; at every hop the holder adds its queries' contribution, and
after c hops the block and its gradients are back home.  Only the order of the
sums differs from :func:`attention_grad`.
"""
from __future__ import annotations

import numpy as np

from oracle import layout


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        import torch
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def _probs(qh, kh, causal):
    """P (exact softmax weights) and lse of one query head against its KV head."""
    S = qh.shape[0]
    s = qh @ kh.T
    if causal:
        s = np.where(np.arange(S)[None, :] > np.arange(S)[:, None], -np.inf, s)
    M = s.max(axis=1, keepdims=True)
    e = np.exp(s - M)
    L = e.sum(axis=1, keepdims=True)
    return e / L, (M + np.log(L))[:, 0]


def attention_grad(q, k, v, dout, causal: bool, out=None):
    """q, dout [Hq, S, d]; k, v [Hkv, S, d] -> dq [Hq, S, d], dk, dv [Hkv, S, d].

    out: the forward output the backward pass is given (D_i = dout_i . out_i is formed
    from it, as a backward pass does); None takes the exact forward output, which makes
    this the exact gradient."""
    q, k, v, dout = (_f64(x) for x in (q, k, v, dout))
    out_given = None if out is None else _f64(out)
    Hq, S, d = q.shape
    Hkv = k.shape[0]
    g = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(Hq):
        hk = h // g
        P, _ = _probs(q[h], k[hk], causal)
        out = P @ v[hk] if out_given is None else out_given[h]
        dP = dout[h] @ v[hk].T
        D = np.einsum("sd,sd->s", dout[h], out)
        dS = P * (dP - D[:, None])
        dq[h] = dS @ k[hk]
        dk[hk] += dS.T @ q[h]
        dv[hk] += P.T @ dout[h]
    return dq, dk, dv


def grad_abs_sums(q, k, v, dout, causal: bool, out=None):
    """Per entry of dq, dk, dv, the sum of the absolute values of the terms it adds up
    (sum_j |dS_ij| |k_j|, sum_i |dS_ij| |q_i|, sum_i P_ij |dout_i|): the scale against
    which rounding of the summed factors is measured.  out: as for attention_grad."""
    q, k, v, dout = (_f64(x) for x in (q, k, v, dout))
    out_given = None if out is None else _f64(out)
    Hq, S, d = q.shape
    Hkv = k.shape[0]
    g = Hq // Hkv
    aq = np.zeros_like(q)
    ak = np.zeros_like(k)
    av = np.zeros_like(v)
    for h in range(Hq):
        hk = h // g
        P, _ = _probs(q[h], k[hk], causal)
        out = P @ v[hk] if out_given is None else out_given[h]
        dP = dout[h] @ v[hk].T
        D = np.einsum("sd,sd->s", dout[h], out)
        adS = np.abs(P * (dP - D[:, None]))
        aq[h] = adS @ np.abs(k[hk])
        ak[hk] += adS.T @ np.abs(q[h])
        av[hk] += P.T @ np.abs(dout[h])
    return aq, ak, av


def ring_backward(q, k, v, dout, c: int, lay: int, causal: bool, kv_block: int):
    """The ring's backward, hop by hop.  Tensors natural [H, S, d]; returns dq, dk, dv
    natural.  Rank r holds its query rows (layout.rank_positions); the KV block that
    starts on rank s is, at hop h, on rank (s + h) mod c, which adds to the block's
    dK, dV and to its own dQ; messages are kv_block rows of the block."""
    q, k, v, dout = (_f64(x) for x in (q, k, v, dout))
    Hq, S, d = q.shape
    Hkv = k.shape[0]
    g = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    pos = [layout.rank_positions(S, c, lay, r) for r in range(c)]
    for h in range(Hq):
        hk = h // g
        P_full, lse = _probs(q[h], k[hk], causal)   # the forward's weights and lse per row
        D = np.einsum("sd,sd->s", dout[h], P_full @ v[hk])   # dout . out, from the forward's out
        for s in range(c):                           # the KV block of rank s ...
            for hop in range(c):                     # ... visits rank (s + hop) mod c
                r = (s + hop) % c
                qi = pos[r]
                for m0 in range(0, len(pos[s]), kv_block):
                    kj = pos[s][m0:m0 + kv_block]
                    sc = q[h][qi] @ k[hk][kj].T
                    if causal:
                        sc = np.where(kj[None, :] > qi[:, None], -np.inf, sc)
                    P = np.exp(sc - lse[qi][:, None])
                    dP = dout[h][qi] @ v[hk][kj].T
                    dS = P * (dP - D[qi][:, None])
                    dq[h][qi] += dS @ k[hk][kj]
                    dk[hk][kj] += dS.T @ q[h][qi]
                    dv[hk][kj] += P.T @ dout[h][qi]
    return dq, dk, dv


def dq_rows(q, k, v, dout, heads, positions, causal: bool, with_abs: bool = False):
    """dq at selected (query head, natural position) rows only: each row's gradient needs
    only its own row of P (and its own D), so long sequences can be checked row by row.
    with_abs: also return sum_j |dS_ij| |k_j| per entry (as grad_abs_sums)."""
    heads = np.asarray(heads, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    Hq = q.shape[0]
    g = Hq // k.shape[0]
    d = q.shape[2]
    res = np.empty((len(heads), d))
    res_abs = np.empty((len(heads), d))
    for h in np.unique(heads):
        idx = np.nonzero(heads == h)[0]
        qh, kh, vh, doh = (_f64(x[int(hh)]) for x, hh in ((q, h), (k, h // g), (v, h // g), (dout, h)))
        for n in idx:
            i = positions[n]
            n_keys = i + 1 if causal else kh.shape[0]
            s = kh[:n_keys] @ qh[i]
            P = np.exp(s - s.max())
            P /= P.sum()
            D = doh[i] @ (P @ vh[:n_keys])
            dS = P * (vh[:n_keys] @ doh[i] - D)
            res[n] = dS @ kh[:n_keys]
            res_abs[n] = np.abs(dS) @ np.abs(kh[:n_keys])
    return (res, res_abs) if with_abs else res


def dkv_rows(q, k, v, dout, kv_heads, positions, causal: bool, with_abs: bool = False, batch_rows: int = 512):
    """dk and dv at selected (KV head, natural key position) rows only.

    A key's gradients add up over every query row that sees it (rows i >= j when
    causal) in every query head of its group: dk_j = sum_i dS_ij q_i and
    dv_j = sum_i P_ij dout_i.  Each such row needs its own lse and D (its whole row of
    scores), so the cost is set by the earliest selected key: keys near the end of a
    causal sequence are cheap.  with_abs: also return the sums of absolute terms
    sum_i |dS_ij| |q_i| and sum_i P_ij |dout_i| (as grad_abs_sums)."""
    kv_heads = np.asarray(kv_heads, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    Hq, S, d = q.shape
    Hkv = k.shape[0]
    g = Hq // Hkv
    dk = np.zeros((len(kv_heads), d))
    dv = np.zeros((len(kv_heads), d))
    ak = np.zeros((len(kv_heads), d))
    av = np.zeros((len(kv_heads), d))
    for hk in np.unique(kv_heads):
        sel = np.nonzero(kv_heads == hk)[0]
        J = positions[sel]
        kh, vh = _f64(k[int(hk)]), _f64(v[int(hk)])
        i0 = int(J.min()) if causal else 0
        rows = np.arange(i0, S)                       # every row that sees a selected key
        for h in range(int(hk) * g, (int(hk) + 1) * g):
            qh, doh = _f64(q[h]), _f64(dout[h])
            for b0 in range(0, len(rows), batch_rows):
                I = rows[b0:b0 + batch_rows]
                n_keys = int(I.max()) + 1 if causal else S
                s = qh[I] @ kh[:n_keys].T              # the rows' whole score rows
                if causal:
                    s = np.where(np.arange(n_keys)[None, :] > I[:, None], -np.inf, s)
                M = s.max(axis=1, keepdims=True)
                e = np.exp(s - M)
                L = e.sum(axis=1, keepdims=True)
                lse = (M + np.log(L))[:, 0]
                D = np.einsum("id,id->i", doh[I], (e @ vh[:n_keys]) / L)
                sj = qh[I] @ kh[J].T                   # [rows, selected keys]
                if causal:
                    sj = np.where(J[None, :] > I[:, None], -np.inf, sj)
                P = np.exp(sj - lse[:, None])
                dS = P * (doh[I] @ vh[J].T - D[:, None])
                dk[sel] += dS.T @ qh[I]
                dv[sel] += P.T @ doh[I]
                ak[sel] += np.abs(dS).T @ np.abs(qh[I])
                av[sel] += P.T @ np.abs(doh[I])
    return (dk, dv, ak, av) if with_abs else (dk, dv)
