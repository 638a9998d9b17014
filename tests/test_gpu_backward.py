"""Backward pass on the GPU (ringattn_bwd, through the C ABI) against the float64 oracle.

Both sides get the same seeded bf16 q, k, v, dout; the GPU also gets the forward's out
and lse as the oracle computes them (float64 rounded to fp32), so that the comparison
isolates the backward.

Tolerance, derived from the arithmetic: the kernel rounds P (for dV) and dS (for dQ, dK)
to bf16, which keeps 8 significant bits (relative error at most 2^-8), and sums every
product in fp32.  An entry g = sum_n a_n b_n whose factors a_n carry relative error 2^-8
is off by at most 2^-8 * A with A = sum_n |a_n| |b_n| (oracle.backward.grad_abs_sums);
fp32 summation, ex2.approx and the fp32 lse add terms some 10^4 times smaller in
practice.  The test allows 2^-8 * A plus 1e-6 of the largest A of the tensor (entries
whose terms nearly cancel, such as dq of a causal row that sees one key, have A ~ 0 and
only the fp32 error), so it checks each entry at the worst case of the rounding itself:
apart from such entries, the largest error over the cases below is 0.93 of 2^-8 * A
(d = 64 with unscaled scores, rows dominated by one key, where one term's rounding is the
whole error).
"""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import backward as obwd
from tests.gpu_util import dev, f64, natural, rank_major

pytestmark = pytest.mark.gpu

REL = 2.0 ** -8


@pytest.fixture(scope="module")
def ra():
    from online_softmax_attention_zigzag_gb300 import ringattn
    ringattn.lib()
    torch.cuda.set_device(0)
    return ringattn


def _randn(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float32) * scale).to(torch.bfloat16)


def _gpu_bwd(ra, q, k, v, dout, out, lse, c, layout, causal, kv_block):
    Hq, S, d = q.shape
    Hkv = k.shape[0]
    rm = lambda x: rank_major(x, S, c, layout).to(dev())  # noqa: E731
    qd, kd, vd, dod = rm(q), rm(k), rm(v), rm(dout)
    od = rm(out.to(torch.float32))
    ld = rank_major(lse.to(torch.float32), S, c, layout).to(dev())
    dq = torch.full((Hq, S, d), float("nan"), dtype=torch.float32, device=dev())
    dk = torch.full((Hkv, S, d), float("nan"), dtype=torch.float32, device=dev())
    dv = torch.full((Hkv, S, d), float("nan"), dtype=torch.float32, device=dev())
    delta = torch.empty((Hq, S), dtype=torch.float32, device=dev())
    ra.bwd(qd, kd, vd, od, ld, dod, dq, dk, dv, delta, c=c, causal=causal, layout=layout, kv_block=kv_block)
    assert ra.sync_status() == ra.RA_OK
    return tuple(natural(x.cpu(), S, c, layout) for x in (dq, dk, dv))


def _forward_oracle(q, k, v, causal):
    o, l = oatt.full_attention(f64(q), f64(k), f64(v), bool(causal))
    return torch.from_numpy(o), torch.from_numpy(l)


CASES = [
    # Hq, Hkv, S, d, c, layout, causal, q scale
    (4, 2, 1024, 128, 2, 1, 1, 128 ** -0.5),   # GQA, zigzag
    (2, 2, 512, 64, 2, 0, 1, 1.0),             # MHA d = 64, contiguous, unscaled scores
    (3, 1, 768, 128, 3, 1, 0, 128 ** -0.5),    # g = 3, non-causal
    (8, 2, 2048, 128, 4, 1, 1, 128 ** -0.5),   # the 4-rank zigzag GQA shape
    (4, 1, 512, 128, 1, 0, 1, 128 ** -0.5),    # one rank (no ring), one KV head for all queries
    (2, 2, 256, 64, 1, 1, 1, 0.125),           # smallest zigzag: one 128-row tile per chunk
    (8, 1, 1024, 64, 2, 1, 0, 0.125),          # g = 8 (the headline's group size), d = 64, non-causal
    (8, 2, 1024, 128, 4, 0, 1, 128 ** -0.5),   # contiguous chunks over 4 ranks, g = 4
]


@pytest.mark.parametrize("case", CASES)
def test_backward_vs_oracle(ra, case):
    Hq, Hkv, S, d, c, layout, causal, scale = case
    q = _randn((Hq, S, d), 201, scale)
    k, v = _randn((Hkv, S, d), 202), _randn((Hkv, S, d), 203)
    dout = _randn((Hq, S, d), 204)
    out, lse = _forward_oracle(q, k, v, causal)
    got = _gpu_bwd(ra, q, k, v, dout, out, lse, c, layout, causal, S // (c * (2 if layout else 1)))
    want = obwd.attention_grad(f64(q), f64(k), f64(v), f64(dout), bool(causal))
    bound = obwd.grad_abs_sums(f64(q), f64(k), f64(v), f64(dout), bool(causal))
    for name, g, w, a in zip(("dq", "dk", "dv"), got, want, bound):
        g = g.double().numpy()
        assert np.isfinite(g).all(), name
        excess = np.abs(g - w) - REL * a
        assert excess.max() <= 1e-6 * a.max(), (name, float(np.abs(g - w).max()), float(excess.max()))


def test_backward_4096_mha_both_layouts(ra):
    """S=4096, 8 heads, d=64, c=4: contiguous and zigzag give the same gradients up to the
    order of the sums, and both meet the bound against the oracle."""
    Hq = Hkv = 8
    S, d, c = 4096, 64, 4
    q, k, v = _randn((Hq, S, d), 211, 0.125), _randn((Hkv, S, d), 212), _randn((Hkv, S, d), 213)
    dout = _randn((Hq, S, d), 214)
    out, lse = _forward_oracle(q, k, v, 1)
    want = obwd.attention_grad(f64(q), f64(k), f64(v), f64(dout), True)
    bound = obwd.grad_abs_sums(f64(q), f64(k), f64(v), f64(dout), True)
    for layout in (0, 1):
        got = _gpu_bwd(ra, q, k, v, dout, out, lse, c, layout, 1, S // (c * (2 if layout else 1)))
        for name, g, w, a in zip(("dq", "dk", "dv"), got, want, bound):
            excess = np.abs(g.double().numpy() - w) - REL * a
            assert excess.max() <= 1e-6 * a.max(), (layout, name)


def test_backward_32k_sampled_rows_and_dv_column_sums(ra):
    """The 32k GQA zigzag workload.
    * dq on 256 sampled rows against the oracle;
    * dk and dv on 256 sampled (KV head, key) rows among the last 512 keys of the sequence,
      against the oracle (a key's gradient adds up over every later row of its 8 query
      heads, so keys near the end are the ones the oracle can afford at this size);
    * for every KV head the exact identity sum_j dv_j = sum over its query heads and rows
      of dout_i (the softmax weights of a row sum to one), within 2^-8 of sum |dout_i|,
      which reaches every key tile of the dK/dV kernel."""
    from online_softmax_attention_zigzag_gb300.configs import CAUSAL_GQA_S32K as w
    from online_softmax_attention_zigzag_gb300.inputs import make_qkv, sample_rows
    q, k, v = make_qkv(w)
    S, c, L = w.seq, w.c, w.layout
    dout = _randn((w.bhq, S, w.d), 221)
    # forward on the GPU supplies out and lse at this size (the oracle cannot: 1.8e13 FLOP)
    qd, kd, vd = (rank_major(x, S, c, L).to(dev()) for x in (q, k, v))
    od = torch.empty((w.bhq, S, w.d), dtype=torch.float32, device=dev())
    ld = torch.empty((w.bhq, S), dtype=torch.float32, device=dev())
    ra.fwd(qd, kd, vd, od, ld, c=c, causal=1, layout=L, kv_block=w.kv_block)
    dod = rank_major(dout, S, c, L).to(dev())
    dq = torch.empty_like(od)
    dk = torch.empty((w.bhkv, S, w.d), dtype=torch.float32, device=dev())
    dv = torch.empty_like(dk)
    delta = torch.empty_like(ld)
    ra.bwd(qd, kd, vd, od, ld, dod, dq, dk, dv, delta, c=c, causal=1, layout=L, kv_block=w.kv_block)
    assert ra.sync_status() == ra.RA_OK
    dq_n = natural(dq.cpu(), S, c, L)
    hs, ps = sample_rows(w.bhq, S, 256)
    want, a = obwd.dq_rows(q, k, v, dout, hs.numpy(), ps.numpy(), True, with_abs=True)
    got = dq_n[hs, ps].double().numpy()
    excess = np.abs(got - want) - REL * a
    assert excess.max() <= 1e-6 * a.max(), float(excess.max())
    # dk, dv at keys among the last 512 positions (and the very last key of each head)
    kh, kp = sample_rows(w.bhkv, 512, 256, seed=1235)
    kp = kp + (S - 512)
    kh = torch.cat([kh, torch.arange(w.bhkv)])
    kp = torch.cat([kp, torch.full((w.bhkv,), S - 1, dtype=torch.int64)])
    wdk, wdv, adk, adv = obwd.dkv_rows(q, k, v, dout, kh.numpy(), kp.numpy(), True, with_abs=True)
    dk_n, dv_n = natural(dk.cpu(), S, c, L), natural(dv.cpu(), S, c, L)
    for name, g_, w_, a_ in (("dk", dk_n, wdk, adk), ("dv", dv_n, wdv, adv)):
        got = g_[kh, kp].double().numpy()
        excess = np.abs(got - w_) - REL * a_
        assert excess.max() <= 1e-6 * a_.max(), (name, float(excess.max()))
    g = w.hq // w.hkv
    dsum = dv.double().sum(dim=1).cpu()                                  # [Hkv, d]
    want_sum = dout.double().reshape(w.bhkv, g, S, w.d).sum(dim=(1, 2))  # [Hkv, d]
    amass = dout.double().abs().reshape(w.bhkv, g, S, w.d).sum(dim=(1, 2))
    assert ((dsum - want_sum).abs() <= REL * amass).all()


def test_natural_order_helpers_forward_and_backward(ra):
    """ringattn.attention then ringattn.attention_backward (permute, ringattn_fwd /
    ringattn_bwd, permute back) on natural-order tensors, against the oracle."""
    Hq, Hkv, S, d = 4, 2, 1024, 64
    q, k, v = _randn((Hq, S, d), 231, 0.125), _randn((Hkv, S, d), 232), _randn((Hkv, S, d), 233)
    dout = _randn((Hq, S, d), 234)
    kw = dict(c=4, causal=1, layout=1, kv_block=128)
    out, lse = ra.attention(q.to(dev()), k.to(dev()), v.to(dev()), **kw)
    grads = ra.attention_backward(q.to(dev()), k.to(dev()), v.to(dev()), out, lse, dout.to(dev()), **kw)
    assert ra.sync_status() == ra.RA_OK
    # D = dout . out comes from the forward's output on both sides
    args = [f64(x) for x in (q, k, v, dout)]
    o64 = f64(out)
    for name, g, w, a in zip(("dq", "dk", "dv"), grads, obwd.attention_grad(*args, True, out=o64),
                             obwd.grad_abs_sums(*args, True, out=o64)):
        excess = np.abs(g.cpu().double().numpy() - w) - REL * a
        assert excess.max() <= 1e-6 * a.max(), name


def test_natural_order_backward_equals_rank_major(ra):
    """ringattn_bwd_natural (chunk map in the kernels' addressing) gives bitwise the
    gradients of ringattn_bwd on rank-major tensors, for both layouts."""
    Hq, Hkv, S, d, c = 8, 2, 2048, 128, 4
    q, k, v = _randn((Hq, S, d), 241, 128 ** -0.5), _randn((Hkv, S, d), 242), _randn((Hkv, S, d), 243)
    dout = _randn((Hq, S, d), 244)
    out, lse = _forward_oracle(q, k, v, 1)
    for layout in (0, 1):
        kvb = S // (c * (2 if layout else 1))
        want = _gpu_bwd(ra, q, k, v, dout, out, lse, c, layout, 1, kvb)
        dq = torch.empty((Hq, S, d), dtype=torch.float32, device=dev())
        dk = torch.empty((Hkv, S, d), dtype=torch.float32, device=dev())
        dv = torch.empty_like(dk)
        delta = torch.empty((Hq, S), dtype=torch.float32, device=dev())
        ra.bwd(q.to(dev()), k.to(dev()), v.to(dev()), out.to(torch.float32).to(dev()),
               lse.to(torch.float32).to(dev()), dout.to(dev()), dq, dk, dv, delta, c=c, causal=1,
               layout=layout, kv_block=kvb, natural=True)
        assert ra.sync_status() == ra.RA_OK
        for g, w in zip((dq, dk, dv), want):
            assert torch.equal(g.cpu(), w)
