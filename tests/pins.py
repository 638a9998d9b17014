"""Checks that pin the CPU oracle to facts outside itself.

Each ``pin_*`` takes the implementation(s) under test as arguments and raises
AssertionError when a fact fails.  ``test_oracle_pins.py`` runs them on the
oracle; ``test_oracle_mutants.py`` runs them on copies of the oracle with one
planted mistake each and expects a failure, which shows that the pins can see
those mistakes.

Facts used (none of them is the oracle's own code):
* closed forms of softmax attention (q = 0, constant V, first causal row,
  one dominant key);
* a pure-Python brute force over tiny inputs;
* ``torch.nn.functional.scaled_dot_product_attention`` and
  ``torch.logsumexp`` in float64, library routines the oracle does not call;
* the identity the pages state: the ring's online-softmax result equals the
  full-row result ("Ring Attention and Ulysses shard a sequence two different
  ways...", the worked example printing True; "Interrogating parallelism,
  part 5", "How does attention survive being split?");
* the zigzag pairing and the per-rank work counts printed in "Interrogating
  parallelism, part 5", "What breaks the load balance?" (fixtures in
  ``tests/golden/``).
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str) -> list[list[str]]:
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# --------------------------------------------------------------------------- full attention

def brute_force(q, k, v, causal):
    """Pure-Python loops, math.exp only; tiny inputs."""
    Hq, S, d = q.shape
    g = Hq // k.shape[0]
    out = [[[0.0] * d for _ in range(S)] for _ in range(Hq)]
    lse = [[0.0] * S for _ in range(Hq)]
    for h in range(Hq):
        kh = h // g
        for i in range(S):
            keys = [j for j in range(S) if (not causal or j <= i)]
            sc = [sum(float(q[h][i][t]) * float(k[kh][j][t]) for t in range(d)) for j in keys]
            M = max(sc)
            w = [math.exp(s - M) for s in sc]
            L = sum(w)
            for t in range(d):
                out[h][i][t] = sum(w[n] * float(v[kh][j][t]) for n, j in enumerate(keys)) / L
            lse[h][i] = M + math.log(L)
    return np.array(out), np.array(lse)


def pin_full_brute(full_fn):
    for causal in (False, True):
        for (Hq, Hkv, S, d, seed) in ((1, 1, 5, 3, 10), (4, 2, 7, 4, 11), (2, 1, 9, 2, 12)):
            q, k, v = rand((Hq, S, d), seed), rand((Hkv, S, d), seed + 100), rand((Hkv, S, d), seed + 200)
            o, l = full_fn(q, k, v, causal)
            ob, lb = brute_force(q, k, v, causal)
            assert np.abs(o - ob).max() < 1e-12, "out differs from brute force"
            assert np.abs(l - lb).max() < 1e-12, "lse differs from brute force"


def pin_full_vs_torch(full_fn):
    for causal in (False, True):
        for (Hq, Hkv, S, d, seed) in ((2, 2, 33, 8, 1), (8, 2, 40, 16, 2), (4, 1, 17, 5, 3)):
            q, k, v = rand((Hq, S, d), seed), rand((Hkv, S, d), seed + 1), rand((Hkv, S, d), seed + 2)
            o, l = full_fn(q, k, v, causal)
            g = Hq // Hkv
            tq = torch.from_numpy(q)
            tk = torch.from_numpy(k).repeat_interleave(g, dim=0)
            tv = torch.from_numpy(v).repeat_interleave(g, dim=0)
            to = torch.nn.functional.scaled_dot_product_attention(
                tq[None], tk[None], tv[None], is_causal=causal, scale=1.0)[0]
            sc = tq @ tk.transpose(-1, -2)
            if causal:
                sc = sc.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
            tl = torch.logsumexp(sc, dim=-1)
            assert np.abs(o - to.numpy()).max() < 1e-10, "out differs from torch SDPA"
            assert np.abs(l - tl.numpy()).max() < 1e-10, "lse differs from torch.logsumexp"


def pin_full_closed_forms(full_fn):
    S, d = 11, 6
    k, v = rand((1, S, d), 21), rand((1, S, d), 22)
    # q = 0: uniform weights over the visible keys
    for causal in (False, True):
        o, l = full_fn(np.zeros((1, S, d)), k, v, causal)
        for i in range(S):
            n = i + 1 if causal else S
            assert np.abs(o[0, i] - v[0, :n].mean(axis=0)).max() < 1e-12, "q=0 is not the mean of V"
            assert abs(l[0, i] - math.log(n)) < 1e-12, "q=0 lse is not ln|A(i)|"
    # constant V: output is that constant whatever the scores
    q = rand((1, S, d), 23)
    for causal in (False, True):
        o, _ = full_fn(q, k, np.full((1, S, d), 0.375), causal)
        assert np.abs(o - 0.375).max() < 1e-12, "constant V not reproduced"
    # first causal row sees only key 0
    o, l = full_fn(q, k, v, True)
    assert np.abs(o[0, 0] - v[0, 0]).max() < 1e-12, "causal row 0 is not v_0"
    assert abs(l[0, 0] - float(q[0, 0] @ k[0, 0])) < 1e-12, "causal row 0 lse is not q0.k0"
    # one dominant key: q along k_j with a score 60 above every other
    kk = np.zeros((1, S, d)); kk[0, :, 0] = 1.0; kk[0, 7, 0] = 61.0
    qq = np.zeros((1, S, d)); qq[0, :, 0] = 1.0
    o, l = full_fn(qq, kk, v, False)
    assert np.abs(o[0] - v[0, 7][None, :]).max() < 2 * S * math.exp(-60) * np.abs(v).max() + 1e-15, \
        "dominant key does not dominate"


# --------------------------------------------------------------------------- ring simulation

def pin_ring_identity(ring_fn, full_fn):
    cases = [
        # (Hq, Hkv, S, d, c, layout, causal, kv_block)
        (1, 1, 12, 8, 3, 0, False, 4),
        (2, 1, 24, 5, 3, 1, True, 2),
        (4, 2, 32, 4, 4, 1, True, 4),
        (2, 2, 32, 4, 4, 0, True, 8),
        (3, 3, 16, 3, 2, 1, False, 1),
        (2, 1, 40, 6, 5, 0, True, 8),
        (1, 1, 20, 3, 1, 0, True, 5),
    ]
    for (Hq, Hkv, S, d, c, layout, causal, kvb) in cases:
        q, k, v = rand((Hq, S, d), S + c), rand((Hkv, S, d), S + c + 1), rand((Hkv, S, d), S + c + 2)
        o, l = ring_fn(q, k, v, c, layout, causal, kvb)
        of, lf = full_fn(q, k, v, causal)
        assert np.abs(o - of).max() < 1e-12, f"ring out != full out for {(c, layout, causal, kvb)}"
        assert np.abs(l - lf).max() < 1e-12, f"ring lse != full lse for {(c, layout, causal, kvb)}"


def pin_worked_example(ring_fn, full_fn):
    g = {r[0]: r[1] for r in read_golden("ring_worked_example.txt")}
    n_q, d, n_kv, blocks = int(g["q_rows"]), int(g["d"]), int(g["kv_rows"]), int(g["blocks"])
    atol = float(g["atol"])
    expected = g["allclose"] == "True"
    # the page's 4x8 q is rank 0's query chunk of a 12-row sequence cut into 3 ring blocks
    q = rand((1, n_kv, d), 5)
    k, v = rand((1, n_kv, d), 6), rand((1, n_kv, d), 7)
    o, _ = ring_fn(q, k, v, blocks, 0, False, n_kv // blocks)
    of, _ = full_fn(q, k, v, False)
    assert np.allclose(of[0, :n_q], o[0, :n_q], atol=atol) == expected


def pin_hop_partials(hop_fn, merge_fn, full_fn):
    """Merging every ring message's partial, in ring order, gives the full result."""
    for (Hq, Hkv, S, d, c, layout, causal, kvb) in ((2, 1, 24, 4, 3, 1, True, 2),
                                                   (1, 1, 16, 3, 4, 0, True, 4),
                                                   (2, 2, 16, 5, 2, 1, False, 4)):
        q, k, v = rand((Hq, S, d), 41), rand((Hkv, S, d), 42), rand((Hkv, S, d), 43)
        o = np.zeros((Hq, S, d)); l = np.full((Hq, S), -np.inf)
        per_hop = (S // c) // kvb
        for hop in range(c):
            for sub in range(per_hop):
                op, lp = hop_fn(q, k, v, c, layout, causal, kvb, hop, sub)
                o, l = merge_fn(o, l, op, lp)
        of, lf = full_fn(q, k, v, causal)
        assert np.abs(o - of).max() < 1e-12 and np.abs(l - lf).max() < 1e-12, "hop partials do not merge to full"


# --------------------------------------------------------------------------- layout and work

def pin_zigzag_golden(rank_chunks_fn):
    rows = read_golden("zigzag_pairing_c8.txt")
    for r, a, b in rows:
        assert list(rank_chunks_fn(8, 1, int(r))) == [int(a), int(b)], f"rank {r} pairing"
    for r in range(8):
        assert list(rank_chunks_fn(8, 0, r)) == [r]


def pin_layout_bijection(order_fn):
    for (S, c, layout) in ((16, 2, 1), (24, 3, 1), (12, 3, 0), (64, 4, 1), (10, 5, 0)):
        perm = np.asarray(order_fn(S, c, layout))
        assert sorted(perm.tolist()) == list(range(S)), "not a permutation of the positions"
        if layout == 0:
            assert perm.tolist() == list(range(S)), "contiguous must be the identity"


def pin_work_golden(work_fn):
    rows = read_golden("causal_work_units_c8.txt")
    S = 16 * 64
    uc, _, _ = work_fn(S, 8, True, 0, 32)
    uz, _, _ = work_fn(S, 8, True, 1, 32)
    for r, cu, zu in rows:
        assert uc[int(r)] == int(cu) and uz[int(r)] == int(zu), f"rank {r} units"
    assert uc[-1] == 8 * uc[0], "contiguous spread is not c-fold"


def pin_work_closed_forms(work_fn):
    for (S, c) in ((1024, 8), (4096, 4), (96, 3)):
        n, m = S // c, S // (2 * c)
        _, pc, _ = work_fn(S, c, True, 0, 32)
        _, pz, _ = work_fn(S, c, True, 1, 32)
        for i in range(c):
            assert pc[i] == i * n * n + n * (n + 1) // 2, "contiguous pairs closed form"
            assert pz[i] == (2 * c - 1) * m * m + m * (m + 1), "zigzag pairs closed form"
        assert pc.sum() == S * (S + 1) // 2 and pz.sum() == S * (S + 1) // 2
    # tiles by brute force over (query, key) pairs on a small case
    S, c, tile = 48, 3, 4
    for layout in (0, 1):
        _, _, t = work_fn(S, c, True, layout, tile)
        from oracle.layout import rank_positions  # positions only, to enumerate pairs
        nch = c * (2 if layout else 1)
        m = S // nch
        for r in range(c):
            pos = rank_positions(S, c, layout, r)
            cnt = 0
            for t0 in range(0, len(pos), tile):
                qs = pos[t0:t0 + tile]
                for kc in range(nch):
                    for k0 in range(kc * m, kc * m + m, tile):
                        ks = range(k0, min(k0 + tile, kc * m + m))
                        cnt += any(kk <= qq for qq in qs for kk in ks)
            assert t[r] == cnt, "tile count"


# --------------------------------------------------------------------------- merge

def pin_merge(merge_fn, full_fn):
    S, d = 14, 5
    q, k, v = rand((1, S, d), 31), rand((1, S, d), 32), rand((1, S, d), 33)
    split = np.array([0, 3, 4, 8, 11, 12])
    rest = np.setdiff1d(np.arange(S), split)
    oa, la = full_fn(q, k[:, split], v[:, split], False)
    ob, lb = full_fn(q, k[:, rest], v[:, rest], False)
    om, lm = merge_fn(oa, la, ob, lb)
    of, lf = full_fn(q, k, v, False)
    assert np.abs(om - of).max() < 1e-12 and np.abs(lm - lf).max() < 1e-12, "merge is not exact"
    om2, lm2 = merge_fn(ob, lb, oa, la)
    assert np.abs(om2 - om).max() < 1e-12 and np.abs(lm2 - lm).max() < 1e-12, "merge not symmetric"
    ninf = np.full_like(la, -np.inf)
    oe, le = merge_fn(oa, la, np.zeros_like(oa), ninf)
    assert np.abs(oe - oa).max() == 0.0 and np.abs(le - la).max() == 0.0, "-inf partial not neutral"
    oz, lz = merge_fn(np.zeros_like(oa), ninf, np.zeros_like(oa), ninf)
    assert np.all(oz == 0.0) and np.all(np.isneginf(lz)), "two empty partials"


# --------------------------------------------------------------------------- document mask

def _segments(doc):
    """[start, end) of every run of equal ids."""
    doc = list(doc)
    segs, a = [], 0
    for i in range(1, len(doc) + 1):
        if i == len(doc) or doc[i] != doc[a]:
            segs.append((a, i))
            a = i
    return segs


def brute_force_doc(q, k, v, doc):
    """Pure-Python loops: keys j <= i of i's document, math.exp only; tiny inputs."""
    Hq, S, d = q.shape
    g = Hq // k.shape[0]
    out = np.zeros((Hq, S, d))
    lse = np.zeros((Hq, S))
    for h in range(Hq):
        kh = h // g
        for i in range(S):
            keys = [j for j in range(i + 1) if doc[j] == doc[i]]
            sc = [sum(float(q[h][i][t]) * float(k[kh][j][t]) for t in range(d)) for j in keys]
            M = max(sc)
            w = [math.exp(s - M) for s in sc]
            L = sum(w)
            for t in range(d):
                out[h][i][t] = sum(w[n] * float(v[kh][j][t]) for n, j in enumerate(keys)) / L
            lse[h][i] = M + math.log(L)
    return out, lse


def pin_doc_brute(doc_fn):
    for (Hq, Hkv, d, doc, seed) in ((2, 1, 3, [0, 0, 0, 1, 1, 2, 3, 3, 3, 3], 70),
                                   (4, 2, 4, [5, 5, 6, 7, 7, 7, 7, 9], 71),
                                   (1, 1, 2, [0, 1, 2, 3, 4], 72)):
        S = len(doc)
        q, k, v = rand((Hq, S, d), seed), rand((Hkv, S, d), seed + 100), rand((Hkv, S, d), seed + 200)
        o, l = doc_fn(q, k, v, np.array(doc))
        ob, lb = brute_force_doc(q, k, v, doc)
        assert np.abs(o - ob).max() < 1e-12, "document-masked out differs from brute force"
        assert np.abs(l - lb).max() < 1e-12, "document-masked lse differs from brute force"


def pin_doc_segments_vs_torch(doc_fn):
    """Each document on its own is plain causal attention (torch SDPA and logsumexp on the
    document's slice): nothing leaks across a boundary and the diagonal is kept."""
    rng = np.random.default_rng(73)
    lens = [1, 7, 2, 33, 1, 1, 20, 64, 3, 18]
    doc = np.repeat(np.arange(len(lens)) * 3 + 2, lens)        # ids need only be equal within a document
    S = len(doc)
    Hq, Hkv, d = 4, 2, 8
    q, k, v = rng.standard_normal((Hq, S, d)), rng.standard_normal((Hkv, S, d)), rng.standard_normal((Hkv, S, d))
    o, l = doc_fn(q, k, v, doc)
    tk = torch.from_numpy(k).repeat_interleave(Hq // Hkv, dim=0)
    tv = torch.from_numpy(v).repeat_interleave(Hq // Hkv, dim=0)
    tq = torch.from_numpy(q)
    for a, b in _segments(doc):
        n = b - a
        to = torch.nn.functional.scaled_dot_product_attention(
            tq[None, :, a:b], tk[None, :, a:b], tv[None, :, a:b], is_causal=True, scale=1.0)[0]
        sc = (tq[:, a:b] @ tk[:, a:b].transpose(-1, -2)).masked_fill(
            torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
        tl = torch.logsumexp(sc, dim=-1)
        assert np.abs(o[:, a:b] - to.numpy()).max() < 1e-10, "document slice differs from torch SDPA"
        assert np.abs(l[:, a:b] - tl.numpy()).max() < 1e-10, "document slice lse differs from logsumexp"


def pin_doc_closed_forms(doc_fn):
    S, d = 12, 5
    q, k, v = rand((1, S, d), 74), rand((1, S, d), 75), rand((1, S, d), 76)
    # every token its own document: it sees only itself
    o, l = doc_fn(q, k, v, np.arange(S))
    assert np.abs(o[0] - v[0]).max() < 1e-12, "single-token document is not v_i"
    assert np.abs(l[0] - np.einsum("sd,sd->s", q[0], k[0])).max() < 1e-12, "single-token lse is not q_i.k_i"
    # q = 0: the mean of V over [start of i's document, i], lse = ln of that count
    doc = np.array([0, 0, 0, 0, 1, 1, 2, 2, 2, 2, 2, 3])
    o, l = doc_fn(np.zeros((1, S, d)), k, v, doc)
    for a, b in _segments(doc):
        for i in range(a, b):
            assert np.abs(o[0, i] - v[0, a:i + 1].mean(axis=0)).max() < 1e-12, "q=0 is not the in-document mean"
            assert abs(l[0, i] - math.log(i - a + 1)) < 1e-12, "q=0 lse is not ln(i - start + 1)"


def pin_doc_pairs(pairs_fn):
    assert pairs_fn(np.arange(9)) == 9
    assert pairs_fn(np.zeros(10, dtype=np.int64)) == 55
    lens = [3, 1, 8, 2]
    assert pairs_fn(np.repeat(np.arange(4), lens)) == sum(n * (n + 1) // 2 for n in lens)


# --------------------------------------------------------------------------- Ulysses relayout

def _positions_by_hand(S, c, lay, r):
    """Natural positions of rank r's tokens in local order, restated from the pages'
    chunking ("What breaks the load balance?") with plain Python ranges."""
    nch = 2 * c if lay == 1 else c
    m = S // nch
    chunks = [r, 2 * c - 1 - r] if lay == 1 else [r]
    return [ch * m + i for ch in chunks for i in range(m)]


def pin_ulysses_relayout(to_heads_fn, to_seq_fn):
    """Sequence-sharded -> head-sharded moves token p, head h of the sequence to
    position p of head h on the rank that keeps h ("Ulysses: an all-to-all relayout
    instead of a rotation"); the inverse brings every value home.  Checked element by
    element with loops, on shards cut from a natural tensor by hand."""
    for (S, H, c, lay, row) in ((12, 4, 2, 1, 3), (12, 6, 3, 0, 2), (16, 4, 4, 1, 1), (8, 3, 1, 0, 2)):
        X = rand((S, H, row), S * 7 + H + c)
        shards = [X[_positions_by_hand(S, c, lay, r)] for r in range(c)]
        heads_of = lambda r: np.arange(r * (H // c), (r + 1) * (H // c))  # noqa: E731
        parts = to_heads_fn(shards, heads_of, S, c, lay)
        assert len(parts) == c
        for r in range(c):
            hs = list(heads_of(r))
            assert parts[r].shape == (len(hs), S, row), "head shard has the wrong shape"
            for i, h in enumerate(hs):
                for p in range(S):
                    assert np.array_equal(parts[r][i, p], X[p, h]), "a value landed in the wrong place"
        back = to_seq_fn(parts, heads_of, H, S, c, lay)
        for r in range(c):
            assert np.array_equal(back[r], shards[r]), "the inverse relayout does not restore the shards"


def pin_ulysses_attention(ulysses_fn):
    """Ulysses gives plain attention (torch SDPA, float64) at every token and head, in
    the sequence-sharded layout, for MHA, GQA and GQA with more ranks than KV heads."""
    cases = [
        # Hq, Hkv, S, d, c, layout, causal
        (4, 4, 16, 5, 2, 1, True),
        (4, 2, 24, 3, 2, 0, True),
        (4, 1, 16, 4, 4, 1, True),
        (6, 3, 12, 2, 3, 0, False),
    ]
    for (Hq, Hkv, S, d, c, lay, causal) in cases:
        seed = Hq * 100 + S + c
        q, k, v = rand((Hq, S, d), seed), rand((Hkv, S, d), seed + 1), rand((Hkv, S, d), seed + 2)
        g = Hq // Hkv
        tq = torch.from_numpy(q)
        tk = torch.from_numpy(k).repeat_interleave(g, dim=0)
        tv = torch.from_numpy(v).repeat_interleave(g, dim=0)
        to = torch.nn.functional.scaled_dot_product_attention(tq[None], tk[None], tv[None], is_causal=causal,
                                                              scale=1.0)[0].numpy()
        sc = tq @ tk.transpose(-1, -2)
        if causal:
            sc = sc.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
        tl = torch.logsumexp(sc, dim=-1).numpy()
        order = [p for r in range(c) for p in _positions_by_hand(S, c, lay, r)]
        seq = lambda x: np.ascontiguousarray(np.swapaxes(x, 0, 1)[order])  # noqa: E731  [S, H, d]
        o, l = ulysses_fn(seq(q), seq(k), seq(v), c, lay, causal)
        assert o.shape == (S, Hq, d) and l.shape == (S, Hq)
        assert np.abs(o - seq(to)).max() < 1e-10, "Ulysses out differs from attention"
        assert np.abs(l - tl.T[order]).max() < 1e-10, "Ulysses lse differs from logsumexp"


# --------------------------------------------------------------------------- backward

def _torch_grads(q, k, v, dout, causal):
    """float64 autograd through torch SDPA (scale 1, GQA by repeating KV heads)."""
    g = q.shape[0] // k.shape[0]
    tq, tk, tv = (torch.from_numpy(np.array(x)).requires_grad_(True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(
        tq[None], tk.repeat_interleave(g, dim=0)[None], tv.repeat_interleave(g, dim=0)[None],
        is_causal=causal, scale=1.0)[0]
    o.backward(torch.from_numpy(np.array(dout)))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


def pin_grad_vs_autograd(grad_fn):
    for causal in (False, True):
        for (Hq, Hkv, S, d, seed) in ((2, 2, 19, 4, 31), (8, 2, 24, 8, 32), (3, 1, 9, 5, 33)):
            q, k, v = rand((Hq, S, d), seed), rand((Hkv, S, d), seed + 1), rand((Hkv, S, d), seed + 2)
            do = rand((Hq, S, d), seed + 3)
            got = grad_fn(q, k, v, do, causal)
            want = _torch_grads(q, k, v, do, causal)
            for name, a, b in zip(("dq", "dk", "dv"), got, want):
                assert np.abs(a - b).max() < 1e-10, f"{name} differs from torch autograd"


def pin_grad_finite_differences(grad_fn):
    """Central differences of sum(out * dout), the forward done by the pure-Python brute
    force, on a tiny GQA case."""
    Hq, Hkv, S, d = 2, 1, 5, 3
    q, k, v, do = rand((Hq, S, d), 41), rand((Hkv, S, d), 42), rand((Hkv, S, d), 43), rand((Hq, S, d), 44)
    for causal in (False, True):
        dq, dk, dv = grad_fn(q, k, v, do, causal)

        def loss(qq, kk, vv):
            o, _ = brute_force(qq, kk, vv, causal)
            return float((o * do).sum())

        eps = 1e-6
        for name, x, gx in (("dq", q, dq), ("dk", k, dk), ("dv", v, dv)):
            for idx in np.ndindex(*x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += eps
                xm[idx] -= eps
                args_p = [xp if y is x else y for y in (q, k, v)]
                args_m = [xm if y is x else y for y in (q, k, v)]
                fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
                assert abs(fd - gx[idx]) < 1e-7, f"{name}{idx} differs from finite differences"


def pin_grad_closed_forms(grad_fn):
    Hq, Hkv, S, d = 2, 1, 10, 4
    q, k, v, do = rand((Hq, S, d), 51), rand((Hkv, S, d), 52), rand((Hkv, S, d), 53), rand((Hq, S, d), 54)
    for causal in (False, True):
        # no gradient flowing in: nothing flows out
        for gx in grad_fn(q, k, v, np.zeros_like(do), causal):
            assert np.abs(gx).max() == 0.0, "dout = 0 must give zero gradients"
        # the same value at every key: out does not depend on the scores
        dq, dk, dv = grad_fn(q, k, np.tile(v[:, :1], (1, S, 1)), do, causal)
        assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12, "constant V must give dq = dk = 0"
        # uniform weights (q = 0): dv_j = sum over the rows that see j of dout_i / |A(i)|
        _, _, dv = grad_fn(np.zeros_like(q), k, v, do, causal)
        for j in range(S):
            rows = range(j, S) if causal else range(S)
            want = sum(do[h, i] / ((i + 1) if causal else S) for h in range(Hq) for i in rows)
            assert np.abs(dv[0, j] - want).max() < 1e-12, "q = 0 dv is not the weighted dout sum"
    # causal row 0 sees one key with weight 1: its dq is exactly zero
    dq, _, _ = grad_fn(q, k, v, do, True)
    assert np.abs(dq[:, 0]).max() < 1e-12, "causal row 0 must have dq = 0"


def pin_ring_backward(ring_grad_fn, grad_fn):
    cases = [
        # (Hq, Hkv, S, d, c, layout, causal, kv_block)
        (2, 2, 16, 4, 2, 1, True, 2), (4, 2, 24, 3, 3, 1, True, 4), (2, 1, 12, 5, 3, 0, False, 2),
        (2, 2, 16, 4, 4, 0, True, 4), (4, 4, 32, 2, 2, 1, False, 8),
    ]
    for (Hq, Hkv, S, d, c, lay, causal, kvb) in cases:
        seed = S + c
        q, k, v = rand((Hq, S, d), seed), rand((Hkv, S, d), seed + 1), rand((Hkv, S, d), seed + 2)
        do = rand((Hq, S, d), seed + 3)
        for a, b in zip(ring_grad_fn(q, k, v, do, c, lay, causal, kvb), grad_fn(q, k, v, do, causal)):
            assert np.abs(a - b).max() < 1e-12, "ring backward differs from the full gradient"


def brute_abs_sums(q, k, v, dout, causal):
    """Pure-Python loops (math.exp only) over every term of every gradient entry:
    sum_j |dS_ij| |k_jt| for dq, sum_i |dS_ij| |q_it| for dk (summed over the query heads
    of a KV head), sum_i P_ij |dout_it| for dv; tiny inputs."""
    Hq, S, d = len(q), len(q[0]), len(q[0][0])
    Hkv = len(k)
    g = Hq // Hkv
    aq = [[[0.0] * d for _ in range(S)] for _ in range(Hq)]
    ak = [[[0.0] * d for _ in range(S)] for _ in range(Hkv)]
    av = [[[0.0] * d for _ in range(S)] for _ in range(Hkv)]
    for h in range(Hq):
        hk = h // g
        for i in range(S):
            keys = [j for j in range(S) if (not causal or j <= i)]
            sc = {j: sum(float(q[h][i][t]) * float(k[hk][j][t]) for t in range(d)) for j in keys}
            M = max(sc.values())
            L = sum(math.exp(s - M) for s in sc.values())
            P = {j: math.exp(sc[j] - M) / L for j in keys}
            out = [sum(P[j] * float(v[hk][j][t]) for j in keys) for t in range(d)]
            D = sum(float(dout[h][i][t]) * out[t] for t in range(d))
            for j in keys:
                dP = sum(float(dout[h][i][t]) * float(v[hk][j][t]) for t in range(d))
                dS = P[j] * (dP - D)
                for t in range(d):
                    aq[h][i][t] += abs(dS) * abs(float(k[hk][j][t]))
                    ak[hk][j][t] += abs(dS) * abs(float(q[h][i][t]))
                    av[hk][j][t] += P[j] * abs(float(dout[h][i][t]))
    return np.array(aq), np.array(ak), np.array(av)


def pin_abs_sums(abs_fn, grad_fn):
    """The sums of absolute terms that scale the backward tolerance: against the
    pure-Python brute force, and exactly equal to |dv| when every dout entry is positive
    (then every term of dv_j = sum_i P_ij dout_i is positive)."""
    for causal in (False, True):
        for (Hq, Hkv, S, d, seed) in ((2, 1, 6, 3, 61), (4, 2, 5, 2, 62)):
            q, k, v = rand((Hq, S, d), seed), rand((Hkv, S, d), seed + 1), rand((Hkv, S, d), seed + 2)
            do = rand((Hq, S, d), seed + 3)
            got = abs_fn(q, k, v, do, causal)
            want = brute_abs_sums(q, k, v, do, causal)
            for name, a, b in zip(("dq", "dk", "dv"), got, want):
                assert np.abs(a - b).max() < 1e-12, f"abs sums of {name} differ from brute force"
            do_pos = np.abs(do) + 0.1
            _, _, av = abs_fn(q, k, v, do_pos, causal)
            _, _, dv = grad_fn(q, k, v, do_pos, causal)
            assert np.abs(av - dv).max() < 1e-12, "with dout > 0 the dv abs sums must equal dv"


def pin_kv_rows(rows_fn, grad_fn, abs_fn):
    """dk, dv (and their abs sums) at selected key rows equal the whole gradient's rows."""
    for causal in (False, True):
        for (Hq, Hkv, S, d, seed) in ((4, 2, 33, 5, 71), (3, 1, 20, 4, 72)):
            q, k, v = rand((Hq, S, d), seed), rand((Hkv, S, d), seed + 1), rand((Hkv, S, d), seed + 2)
            do = rand((Hq, S, d), seed + 3)
            _, dk, dv = grad_fn(q, k, v, do, causal)
            _, ak, av = abs_fn(q, k, v, do, causal)
            rng = np.random.default_rng(seed)
            hk = rng.integers(0, Hkv, 9)
            pos = np.concatenate([[0, S - 1], rng.integers(0, S, 7)])
            r_dk, r_dv, r_ak, r_av = rows_fn(q, k, v, do, hk, pos, causal, with_abs=True, batch_rows=4)
            for name, a, b in (("dk", r_dk, dk), ("dv", r_dv, dv), ("|dk|", r_ak, ak), ("|dv|", r_av, av)):
                assert np.abs(a - b[hk, pos]).max() < 1e-12, f"{name} rows differ from the whole gradient"
