"""The oracle against facts outside itself (CPU only)."""
import numpy as np
import pytest

from oracle import attention, docmask, layout, merge, ring, work
from tests import pins


def test_full_vs_brute_force():
    pins.pin_full_brute(attention.full_attention)


def test_full_vs_torch_library():
    pins.pin_full_vs_torch(attention.full_attention)


def test_full_closed_forms():
    pins.pin_full_closed_forms(attention.full_attention)


def test_full_rows_matches_library():
    # the row-subset form against torch's SDPA on selected rows
    import torch
    rng = np.random.default_rng(3)
    Hq, Hkv, S, d = 4, 2, 300, 8
    q, k, v = rng.standard_normal((Hq, S, d)), rng.standard_normal((Hkv, S, d)), rng.standard_normal((Hkv, S, d))
    heads = np.array([0, 0, 1, 3, 3, 2])
    posn = np.array([0, 299, 17, 150, 151, 64])
    for causal in (False, True):
        o, l = attention.full_attention_rows(q, k, v, heads, posn, causal, batch_rows=2)
        tk = torch.from_numpy(k).repeat_interleave(2, 0)
        tv = torch.from_numpy(v).repeat_interleave(2, 0)
        to = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None], tk[None], tv[None], is_causal=causal, scale=1.0)[0]
        assert np.abs(o - to.numpy()[heads, posn]).max() < 1e-10


def test_ring_equals_full():
    pins.pin_ring_identity(ring.ring_attention, attention.full_attention)


def test_worked_example():
    pins.pin_worked_example(ring.ring_attention, attention.full_attention)


def test_hop_partials_merge_to_full():
    pins.pin_hop_partials(ring.ring_hop_partial, merge.merge, attention.full_attention)


def test_merge_exact():
    pins.pin_merge(merge.merge, attention.full_attention)


def test_zigzag_pairing_golden():
    pins.pin_zigzag_golden(layout.rank_chunks)


def test_layout_bijection_and_inverse():
    pins.pin_layout_bijection(layout.rank_major_order)
    x = np.arange(2 * 48 * 3).reshape(2, 48, 3)
    for (c, lay) in ((3, 0), (3, 1), (4, 1), (1, 1)):
        y = layout.to_rank_major(x, 48, c, lay)
        assert np.array_equal(layout.from_rank_major(y, 48, c, lay), x)


def test_work_golden():
    pins.pin_work_golden(work.rank_work)


def test_work_closed_forms():
    pins.pin_work_closed_forms(work.rank_work)


def test_ring_schedule_covers_each_key_once():
    for (S, c, lay, kvb) in ((32, 4, 1, 2), (24, 3, 0, 4), (16, 1, 1, 8)):
        for r in range(c):
            msgs = ring.ring_schedule(S, c, lay, r, kvb)
            allk = np.sort(np.concatenate(msgs))
            assert np.array_equal(allk, np.arange(S))
            # hop 0 is the rank's own block (no communication on the first round)
            own = layout.rank_positions(S, c, lay, r)
            assert np.array_equal(np.concatenate(msgs[: len(own) // kvb]), own)


def test_doc_mask_vs_brute_force():
    pins.pin_doc_brute(docmask.doc_attention)


def test_doc_mask_each_document_is_causal_attention():
    pins.pin_doc_segments_vs_torch(docmask.doc_attention)


def test_doc_mask_closed_forms():
    pins.pin_doc_closed_forms(docmask.doc_attention)


def test_doc_mask_rows_match_whole():
    rng = np.random.default_rng(77)
    Hq, Hkv, S, d = 4, 2, 90, 6
    q, k, v = rng.standard_normal((Hq, S, d)), rng.standard_normal((Hkv, S, d)), rng.standard_normal((Hkv, S, d))
    doc = np.repeat(np.arange(6), [10, 1, 30, 4, 40, 5])
    o, l = docmask.doc_attention(q, k, v, doc)
    heads, posn = np.array([0, 1, 3, 3, 2]), np.array([0, 10, 11, 89, 45])
    ro, rl = docmask.doc_attention_rows(q, k, v, doc, heads, posn, batch_rows=2)
    assert np.abs(ro - o[heads, posn]).max() < 1e-12 and np.abs(rl - l[heads, posn]).max() < 1e-12


def test_doc_pairs():
    pins.pin_doc_pairs(docmask.doc_pairs)


def test_ulysses_relayout_moves_every_value_home():
    from oracle import ulysses
    pins.pin_ulysses_relayout(ulysses.seq_to_heads, ulysses.heads_to_seq)


def test_ulysses_attention_is_attention():
    from oracle import ulysses
    pins.pin_ulysses_attention(ulysses.ulysses_attention)


def test_ulysses_kv_heads_replicate_when_ranks_outnumber_them():
    from oracle import ulysses
    # 8 query heads over 2 KV heads on 4 ranks: ranks 0-1 need KV head 0, ranks 2-3 KV head 1
    assert [list(ulysses.kv_heads(8, 2, 4, r)) for r in range(4)] == [[0], [0], [1], [1]]
    assert [list(ulysses.kv_heads(8, 4, 2, r)) for r in range(2)] == [[0, 1], [2, 3]]


def test_backward_vs_torch_autograd():
    from oracle import backward
    pins.pin_grad_vs_autograd(backward.attention_grad)


def test_backward_vs_finite_differences():
    from oracle import backward
    pins.pin_grad_finite_differences(backward.attention_grad)


def test_backward_closed_forms():
    from oracle import backward
    pins.pin_grad_closed_forms(backward.attention_grad)


def test_ring_backward_is_the_gradient():
    from oracle import backward
    pins.pin_ring_backward(backward.ring_backward, backward.attention_grad)


def test_backward_abs_sums_bound_the_gradients():
    from oracle import backward
    rng = np.random.default_rng(5)
    q, k, v, do = (rng.standard_normal(s) for s in ((4, 20, 3), (2, 20, 3), (2, 20, 3), (4, 20, 3)))
    for causal in (False, True):
        for g, a in zip(backward.attention_grad(q, k, v, do, causal), backward.grad_abs_sums(q, k, v, do, causal)):
            assert (np.abs(g) <= a + 1e-12).all() and (a >= 0).all()


def test_backward_abs_sums_vs_brute_force():
    from oracle import backward
    pins.pin_abs_sums(backward.grad_abs_sums, backward.attention_grad)


def test_backward_kv_rows_match_whole():
    from oracle import backward
    pins.pin_kv_rows(backward.dkv_rows, backward.attention_grad, backward.grad_abs_sums)


def test_backward_dq_rows_match_whole():
    from oracle import backward
    rng = np.random.default_rng(9)
    q, k, v, do = (rng.standard_normal(s) for s in ((4, 30, 5), (2, 30, 5), (2, 30, 5), (4, 30, 5)))
    heads, posn = np.array([0, 3, 1, 2, 3]), np.array([0, 29, 7, 15, 1])
    for causal in (False, True):
        dq, _, _ = backward.attention_grad(q, k, v, do, causal)
        assert np.abs(backward.dq_rows(q, k, v, do, heads, posn, causal) - dq[heads, posn]).max() < 1e-12
        aq, _, _ = backward.grad_abs_sums(q, k, v, do, causal)
        _, ra_ = backward.dq_rows(q, k, v, do, heads, posn, causal, with_abs=True)
        assert np.abs(ra_ - aq[heads, posn]).max() < 1e-12


def test_backward_given_out():
    """Given the exact forward output, D is the same and so is the gradient; given a
    perturbed one, only dq and dk move, and by exactly -P_ij (dout_i . delta_i) terms."""
    from oracle import attention, backward
    rng = np.random.default_rng(11)
    q, k, v, do = (rng.standard_normal(s) for s in ((2, 12, 3), (1, 12, 3), (1, 12, 3), (2, 12, 3)))
    o, _ = attention.full_attention(q, k, v, True)
    for a, b in zip(backward.attention_grad(q, k, v, do, True), backward.attention_grad(q, k, v, do, True, out=o)):
        assert np.abs(a - b).max() < 1e-12
    dlt = rng.standard_normal(o.shape) * 1e-3
    g0 = backward.attention_grad(q, k, v, do, True)
    g1 = backward.attention_grad(q, k, v, do, True, out=o + dlt)
    assert np.abs(g1[2] - g0[2]).max() < 1e-14                       # dv does not use D
    dD = np.einsum("hsd,hsd->hs", do, dlt)                           # change of D per row
    P = np.exp(np.where(np.triu(np.ones((12, 12)), 1) > 0, -np.inf, q @ k[0].T)
               - attention.full_attention(q, k, v, True)[1][..., None])
    want_dq = g0[0] - np.einsum("hij,hi,jd->hid", P, dD, k[0])
    assert np.abs(g1[0] - want_dq).max() < 1e-12
