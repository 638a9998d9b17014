"""Plant one plausible mistake at a time in a copy of the oracle and check
that the pins reject it (CPU only).  The oracle itself is not modified."""
import numpy as np
import pytest

from oracle import attention, layout, merge, ring, work
from tests import pins


# ---------------------------------------------------------------- full attention mutants

def _full(q, k, v, causal, *, off=0, lse_no_max=False, gqa_mod=False, no_norm=False, rev_k=False):
    q = np.asarray(q, float); k = np.asarray(k, float); v = np.asarray(v, float)
    Hq, S, d = q.shape
    Hkv = k.shape[0]
    g = Hq // Hkv
    out = np.empty((Hq, S, v.shape[2])); lse = np.empty((Hq, S))
    for h in range(Hq):
        kh = h % Hkv if gqa_mod else h // g
        kk = k[kh][:, ::-1] if rev_k else k[kh]
        s = q[h] @ kk.T
        if causal:
            s = np.where(np.arange(S)[None, :] > np.arange(S)[:, None] + off, -np.inf, s)
        M = s.max(1)
        e = np.exp(s - M[:, None])
        L = e.sum(1)
        out[h] = (e @ v[kh]) / (1.0 if no_norm else L[:, None])
        lse[h] = (0.0 if lse_no_max else M) + np.log(L)
    return out, lse


FULL_MUTANTS = {
    "mask_off_by_one": dict(off=1),
    "lse_drops_max": dict(lse_no_max=True),
    "gqa_head_map_mod": dict(gqa_mod=True),
    "no_normalisation": dict(no_norm=True),
    "key_features_reversed": dict(rev_k=True),
}


@pytest.mark.parametrize("name", sorted(FULL_MUTANTS))
def test_full_mutant_caught(name):
    kw = FULL_MUTANTS[name]
    fn = lambda q, k, v, causal: _full(q, k, v, causal, **kw)  # noqa: E731
    failures = 0
    for pin in (pins.pin_full_brute, pins.pin_full_vs_torch, pins.pin_full_closed_forms):
        try:
            pin(fn)
        except AssertionError:
            failures += 1
    assert failures > 0, f"mutant {name} passed every pin"


def test_unmutated_copy_passes():
    # the mutant harness with no mutation is a faithful copy: all pins pass
    fn = lambda q, k, v, causal: _full(q, k, v, causal)  # noqa: E731
    pins.pin_full_brute(fn)
    pins.pin_full_vs_torch(fn)
    pins.pin_full_closed_forms(fn)


# ---------------------------------------------------------------- ring mutants

def _ring_rank(q_rows, q_pos, k, v, blocks, causal, *, no_out_corr=False, no_sum_corr=False, flip=False):
    """The oracle's per-rank accumulator (reference max, exponential sum, weighted
    values), with one of its rescaling steps planted wrong."""
    n = q_rows.shape[0]
    ref = np.full(n, -np.inf); tot = np.zeros(n); wsum = np.zeros((n, v.shape[1]))
    for keys in blocks:
        blk = q_rows @ k[keys].T
        if causal:
            blk = np.where(keys[None, :] <= q_pos[:, None], blk, -np.inf)
        nxt = np.maximum(ref, blk.max(axis=1))
        live = nxt > -np.inf
        base = np.where(live, nxt, 0.0)
        with np.errstate(invalid="ignore", over="ignore"):
            step = (base - ref) if flip else (ref - base)
            alpha = np.where(live & (ref > -np.inf), np.exp(step), 0.0)
        w = np.exp(blk - base[:, None])
        w[~live] = 0.0
        tot = (tot if no_sum_corr else alpha * tot) + w.sum(axis=1)
        wsum = (wsum if no_out_corr else alpha[:, None] * wsum) + w @ v[keys]
        ref = nxt
    with np.errstate(divide="ignore", invalid="ignore"):
        return wsum / tot[:, None], ref + np.log(tot)


def _ring(q, k, v, c, lay, causal, kvb, **kw):
    q = np.asarray(q, float); k = np.asarray(k, float); v = np.asarray(v, float)
    Hq, S, d = q.shape
    g = Hq // k.shape[0]
    out = np.zeros((Hq, S, v.shape[2])); lse = np.zeros((Hq, S))
    for h in range(Hq):
        for r in range(c):
            pos = layout.rank_positions(S, c, lay, r)
            o, l = _ring_rank(q[h, pos], pos, k[h // g], v[h // g],
                              ring.ring_schedule(S, c, lay, r, kvb), causal, **kw)
            out[h, pos] = o; lse[h, pos] = l
    return out, lse


RING_MUTANTS = {
    "output_not_rescaled": dict(no_out_corr=True),
    "sum_not_rescaled": dict(no_sum_corr=True),
    "correction_sign_flipped": dict(flip=True),
}


@pytest.mark.parametrize("name", sorted(RING_MUTANTS))
def test_ring_mutant_caught(name):
    kw = RING_MUTANTS[name]
    fn = lambda *a: _ring(*a, **kw)  # noqa: E731
    with pytest.raises(AssertionError):
        pins.pin_ring_identity(fn, attention.full_attention)


def test_ring_copy_passes():
    pins.pin_ring_identity(lambda *a: _ring(*a), attention.full_attention)


# ---------------------------------------------------------------- layout / work / merge mutants

def test_zigzag_pairing_mutant_caught():
    bad = lambda c, lay, r: [r, 2 * c - 2 - r] if lay == 1 else [r]  # noqa: E731
    with pytest.raises(AssertionError):
        pins.pin_zigzag_golden(bad)


def test_work_mutants_caught():
    def shifted(S, c, causal, lay, tile):
        u, p, t = work.rank_work(S, c, causal, lay, tile)
        return (u[::-1] if lay == 0 else u - 1), p, t

    with pytest.raises(AssertionError):
        pins.pin_work_golden(shifted)

    def half_diag(S, c, causal, lay, tile):
        u, p, t = work.rank_work(S, c, causal, lay, tile)
        m = S // (c * (2 if lay else 1))
        return u, p - m // 2, t

    with pytest.raises(AssertionError):
        pins.pin_work_closed_forms(half_diag)


def test_merge_mutants_caught():
    def unnormalised(oa, la, ob, lb):
        o, l = merge.merge(oa, la, ob, lb)
        return o * 1.0001, l

    def lse_sum(oa, la, ob, lb):
        o, _ = merge.merge(oa, la, ob, lb)
        return o, np.maximum(la, lb)

    for fn in (unnormalised, lse_sum):
        with pytest.raises(AssertionError):
            pins.pin_merge(fn, attention.full_attention)


# ---------------------------------------------------------------- document-mask mutants

def _doc(q, k, v, doc, *, leak_earlier=False, no_diag=False, no_causal=False, gqa_mod=False, shift=False):
    q = np.asarray(q, float); k = np.asarray(k, float); v = np.asarray(v, float)
    doc = np.asarray(doc)
    Hq, S, d = q.shape
    Hkv = k.shape[0]
    out = np.empty((Hq, S, v.shape[2])); lse = np.empty((Hq, S))
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    di = doc[np.maximum(np.arange(S) - 1, 0)] if shift else doc
    same = (doc[None, :] <= di[:, None]) if leak_earlier else (doc[None, :] == di[:, None])
    causal = (j < i) if no_diag else (j <= i)
    vis = same if no_causal else (same & causal)
    for h in range(Hq):
        kh = h % Hkv if gqa_mod else h // (Hq // Hkv)
        s = np.where(vis, q[h] @ k[kh].T, -np.inf)
        M = s.max(1)
        e = np.exp(s - M[:, None])
        L = e.sum(1)
        out[h] = (e @ v[kh]) / L[:, None]
        lse[h] = M + np.log(L)
    return out, lse


DOC_MUTANTS = {
    "attends_earlier_documents": dict(leak_earlier=True),
    "drops_the_diagonal": dict(no_diag=True),
    "not_causal_inside_a_document": dict(no_causal=True),
    "gqa_head_map_mod": dict(gqa_mod=True),
    "document_of_previous_token": dict(shift=True),
}


@pytest.mark.parametrize("name", sorted(DOC_MUTANTS))
def test_doc_mutant_caught(name):
    kw = DOC_MUTANTS[name]
    fn = lambda q, k, v, doc: _doc(q, k, v, doc, **kw)  # noqa: E731
    failures = 0
    for pin in (pins.pin_doc_brute, pins.pin_doc_segments_vs_torch, pins.pin_doc_closed_forms):
        try:
            with np.errstate(invalid="ignore", divide="ignore"):
                pin(fn)
        except AssertionError:
            failures += 1
    assert failures > 0, f"mutant {name} passed every pin"


def test_doc_copy_passes():
    fn = lambda q, k, v, doc: _doc(q, k, v, doc)  # noqa: E731
    pins.pin_doc_brute(fn)
    pins.pin_doc_segments_vs_torch(fn)
    pins.pin_doc_closed_forms(fn)


# ---------------------------------------------------------------- Ulysses relayout mutants

def _to_heads(shards, heads_of, S, c, lay, *, local_order=False, contiguous_map=False):
    row = shards[0].shape[2:]
    out = [np.zeros((len(heads_of(r)), S) + row) for r in range(c)]
    for s in range(c):
        if local_order:                 # tokens stored where they sit on the sender, not by position
            pos = np.arange(s * shards[s].shape[0], (s + 1) * shards[s].shape[0])
        else:
            pos = layout.rank_positions(S, c, 0 if contiguous_map else lay, s)
        for r in range(c):
            out[r][:, pos] = np.swapaxes(shards[s][:, heads_of(r)], 0, 1)
    return out


def _to_seq(parts, heads_of, H, S, c, lay):
    from oracle import ulysses
    return ulysses.heads_to_seq(parts, heads_of, H, S, c, lay)


@pytest.mark.parametrize("kw", [dict(local_order=True), dict(contiguous_map=True)])
def test_ulysses_relayout_mutant_caught(kw):
    with pytest.raises(AssertionError):
        pins.pin_ulysses_relayout(lambda *a: _to_heads(*a, **kw), _to_seq)


def test_ulysses_relayout_unmutated_copy_passes():
    pins.pin_ulysses_relayout(_to_heads, _to_seq)


def test_ulysses_attention_mutants_caught():
    from oracle import ulysses

    def wrong_heads(q_seq, k_seq, v_seq, c, lay, causal):
        # every rank takes KV head (rank) instead of the KV heads its query heads use
        q_seq, k_seq, v_seq = (np.asarray(x, float) for x in (q_seq, k_seq, v_seq))
        S, Hq, d = q_seq.shape
        Hkv = k_seq.shape[1]
        out = np.empty((S, Hq, d)); lse = np.empty((S, Hq))
        order = layout.rank_major_order(S, c, lay)
        qn = np.empty_like(q_seq); kn = np.empty_like(k_seq); vn = np.empty_like(v_seq)
        qn[order], kn[order], vn[order] = q_seq, k_seq, v_seq
        for h in range(Hq):
            r = h // (Hq // c)
            o, l = attention.full_attention(qn[:, h][None], kn[:, r % Hkv][None], vn[:, r % Hkv][None], causal)
            out[:, h] = o[0][order]; lse[:, h] = l[0][order]
        return out, lse

    with pytest.raises(AssertionError):
        pins.pin_ulysses_attention(wrong_heads)
    pins.pin_ulysses_attention(ulysses.ulysses_attention)


# ---------------------------------------------------------------- backward mutants

def _grad(q, k, v, dout, causal, *, flip=False, no_delta=False, dk_untransposed=False, overwrite=False):
    from oracle import backward as ob
    q, k, v, dout = (np.asarray(x, float) for x in (q, k, v, dout))
    Hq, S, d = q.shape
    g = Hq // k.shape[0]
    dq = np.zeros_like(q); dk = np.zeros_like(k); dv = np.zeros_like(v)
    for h in range(Hq):
        hk = h // g
        P, _ = ob._probs(q[h], k[hk], causal)
        D = 0.0 if no_delta else np.einsum("sd,sd->s", dout[h], P @ v[hk])[:, None]
        dP = dout[h] @ v[hk].T
        dS = P * ((D - dP) if flip else (dP - D))
        dq[h] = dS @ k[hk]
        t = (dS @ q[h]) if dk_untransposed else (dS.T @ q[h])
        if overwrite:
            dk[hk] = t
            dv[hk] = P.T @ dout[h]
        else:
            dk[hk] += t
            dv[hk] += P.T @ dout[h]
    return dq, dk, dv


GRAD_MUTANTS = {
    "dS_sign_flipped": dict(flip=True),
    "delta_dropped": dict(no_delta=True),
    "dK_not_transposed": dict(dk_untransposed=True),
    "gqa_grads_overwritten": dict(overwrite=True),
}


@pytest.mark.parametrize("name", sorted(GRAD_MUTANTS))
def test_grad_mutant_caught(name):
    kw = GRAD_MUTANTS[name]
    fn = lambda q, k, v, do, causal: _grad(q, k, v, do, causal, **kw)  # noqa: E731
    failures = 0
    for pin in (pins.pin_grad_vs_autograd, pins.pin_grad_closed_forms):
        try:
            pin(fn)
        except AssertionError:
            failures += 1
    assert failures > 0, f"mutant {name} passed every pin"


def test_grad_unmutated_copy_passes():
    fn = lambda q, k, v, do, causal: _grad(q, k, v, do, causal)  # noqa: E731
    pins.pin_grad_vs_autograd(fn)
    pins.pin_grad_closed_forms(fn)


# ---------------------------------------------------------------- abs-sum mutants (backward tolerance scale)

def _abs_sums(q, k, v, dout, causal, *, inflate=1.0, p_for_ds=False, signed_k=False, ak_uses_p=False):
    from oracle import backward as ob
    q, k, v, dout = (np.asarray(x, float) for x in (q, k, v, dout))
    Hq, S, d = q.shape
    g = Hq // k.shape[0]
    aq = np.zeros_like(q); ak = np.zeros_like(k); av = np.zeros_like(v)
    for h in range(Hq):
        hk = h // g
        P, _ = ob._probs(q[h], k[hk], causal)
        D = np.einsum("sd,sd->s", dout[h], P @ v[hk])[:, None]
        adS = np.abs(P * (dout[h] @ v[hk].T - D))
        aq[h] = (P if p_for_ds else adS) @ (k[hk] if signed_k else np.abs(k[hk]))
        ak[hk] += (P if ak_uses_p else adS).T @ np.abs(q[h])
        av[hk] += P.T @ np.abs(dout[h])
    return aq * inflate, ak * inflate, av * inflate


ABS_MUTANTS = {
    "inflated_by_two": dict(inflate=2.0),
    "P_in_place_of_dS_for_dq": dict(p_for_ds=True),
    "k_not_taken_absolute": dict(signed_k=True),
    "P_in_place_of_dS_for_dk": dict(ak_uses_p=True),
}


@pytest.mark.parametrize("name", sorted(ABS_MUTANTS))
def test_abs_sums_mutant_caught(name):
    from oracle import backward
    kw = ABS_MUTANTS[name]
    fn = lambda q, k, v, do, causal: _abs_sums(q, k, v, do, causal, **kw)  # noqa: E731
    with pytest.raises(AssertionError):
        pins.pin_abs_sums(fn, backward.attention_grad)


def test_abs_sums_unmutated_copy_passes():
    from oracle import backward
    pins.pin_abs_sums(lambda q, k, v, do, causal: _abs_sums(q, k, v, do, causal), backward.attention_grad)
