"""Parity of the CUDA path (through the C ABI) with the float64 CPU oracle.

Every test feeds the same seeded inputs to both sides; the oracle never sees a
value the GPU produced except as the thing being checked.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import layout as olay
from oracle import merge as omerge
from oracle import ring as oring
from tests.gpu_util import TOL_BF16_LSE, TOL_BF16_OUT, TOL_F32, dev, f64, max_err, natural, rank_major

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import os

    from online_softmax_attention_zigzag_gb300 import ringattn
    if not os.path.exists(ringattn.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    torch.cuda.set_device(0)
    return ringattn


def _status_ok(ra):
    assert ra.sync_status() == ra.RA_OK


def _randn(shape, seed, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(dtype)


# ------------------------------------------------------------------ permutation (bit-exact)

@pytest.mark.parametrize("S,H,row_bytes,c,layout", [
    (4096, 8, 128, 4, 1), (4096, 8, 128, 4, 0), (96, 3, 3, 3, 1), (96, 3, 4, 3, 1),
    (1024, 2, 512, 8, 1), (48, 5, 6, 2, 1), (2048, 3, 256, 1, 1), (640, 2, 2, 5, 0),
])
def test_permute_bit_exact(ra, S, H, row_bytes, c, layout):
    g = torch.Generator().manual_seed(S + H + row_bytes)
    x = torch.randint(0, 256, (H, S, row_bytes), generator=g, dtype=torch.uint8)
    xd = x.to(dev())
    y = torch.empty_like(xd)
    ra.permute(xd, y, c=c, layout=layout, inverse=0)
    want = olay.to_rank_major(x.numpy(), S, c, layout)
    assert np.array_equal(y.cpu().numpy(), want)
    z = torch.empty_like(xd)
    ra.permute(y, z, c=c, layout=layout, inverse=1)
    assert torch.equal(z.cpu(), x)
    _status_ok(ra)


def test_permute_bf16_and_f32_rows(ra):
    S, c = 1024, 4
    q = _randn((4, S, 64), 3, torch.bfloat16)
    qd = q.to(dev())
    y = torch.empty_like(qd)
    ra.permute(qd, y, c=c, layout=1, inverse=0)
    assert torch.equal(y.cpu(), rank_major(q, S, c, 1))
    lse = _randn((4, S), 4)
    ld = lse.to(dev())
    ly = torch.empty_like(ld)
    ra.permute(ld, ly, c=c, layout=1, inverse=0)
    assert torch.equal(ly.cpu(), rank_major(lse, S, c, 1))


# ------------------------------------------------------------------ merge

@pytest.mark.parametrize("rows,d", [(1000, 128), (333, 64), (17, 5), (64, 8)])
def test_merge_vs_oracle(ra, rows, d):
    oa, ob = _randn((rows, d), 1), _randn((rows, d), 2)
    la, lb = _randn((rows,), 3) * 20, _randn((rows,), 4) * 20
    la[::7] = -np.inf
    lb[::5] = -np.inf
    oa[::7] = float("nan")  # an empty side's o must not leak into the result
    want_o, want_l = omerge.merge(np.nan_to_num(oa.numpy()), la.numpy(), ob.numpy(), lb.numpy())
    od, ld = oa.to(dev()), la.to(dev())
    ra.merge(od, ld, ob.to(dev()), lb.to(dev()))
    assert max_err(od.cpu(), want_o) < 2e-6
    assert max_err(ld.cpu(), want_l) < 2e-5
    _status_ok(ra)


# ------------------------------------------------------------------ fp32 path

def _run_f32(ra, q, k, v, c, layout, causal, kv_block):
    Hq, S, d = q.shape
    qd, kd, vd = (rank_major(x, S, c, layout).to(dev()) for x in (q, k, v))
    o = torch.empty((Hq, S, d), dtype=torch.float32, device=dev())
    l = torch.empty((Hq, S), dtype=torch.float32, device=dev())
    ra.fwd_f32(qd, kd, vd, o, l, c=c, causal=causal, layout=layout, kv_block=kv_block)
    torch.cuda.synchronize()
    return natural(o.cpu(), S, c, layout), natural(l.cpu(), S, c, layout)


def test_f32_worked_example(ra):
    """12 keys in 3 ring blocks of 4, q 4x8 of rank 0 plus the other ranks' rows."""
    from online_softmax_attention_zigzag_gb300.configs import TINY_F32 as w
    from online_softmax_attention_zigzag_gb300.inputs import make_qkv
    q, k, v = make_qkv(w)
    o, l = _run_f32(ra, q, k, v, w.c, w.layout, w.causal, w.kv_block)
    ro, rl = oatt.full_attention(f64(q), f64(k), f64(v), False)
    assert max_err(o, ro) <= TOL_F32 and max_err(l, rl) <= TOL_F32
    # the page's 4x8 query block: rank 0's rows, allclose at atol 1e-6 in float64 terms
    assert np.allclose(f64(o)[0, :4], ro[0, :4], atol=1e-6)
    _status_ok(ra)


F32_CASES = [
    # Hq, Hkv, S, d, c, layout, causal, kv_block
    (1, 1, 12, 8, 3, 0, 0, 1), (1, 1, 12, 8, 3, 0, 1, 2), (2, 1, 24, 5, 3, 1, 1, 2),
    (4, 2, 32, 16, 4, 1, 1, 4), (3, 3, 64, 64, 2, 1, 0, 8), (2, 2, 48, 128, 1, 0, 1, 48),
    (2, 1, 96, 3, 4, 0, 1, 8), (4, 4, 160, 32, 5, 1, 1, 16), (1, 1, 300, 100, 3, 0, 1, 50),
]


@pytest.mark.parametrize("case", F32_CASES)
def test_f32_sweep(ra, case):
    Hq, Hkv, S, d, c, layout, causal, kvb = case
    # q scaled by 1/sqrt(d) keeps scores O(1): the 1e-5 bound is then above fp32's own
    # rounding of a d-term dot product (unscaled d = 128 scores reach ~30, where the
    # accumulation alone can err by ~1e-5)
    q = _randn((Hq, S, d), 11) / d ** 0.5
    k, v = _randn((Hkv, S, d), 12), _randn((Hkv, S, d), 13)
    o, l = _run_f32(ra, q, k, v, c, layout, causal, kvb)
    ro, rl = oatt.full_attention(f64(q), f64(k), f64(v), bool(causal))
    assert max_err(o, ro) <= TOL_F32
    assert max_err(l, rl) <= TOL_F32


@pytest.mark.parametrize("case", [(2, 1, 24, 5, 3, 1, 1, 2), (1, 1, 12, 8, 3, 0, 0, 4), (2, 2, 64, 32, 4, 0, 1, 8)])
def test_f32_hop_partials_and_merge(ra, case):
    Hq, Hkv, S, d, c, layout, causal, kvb = case
    q, k, v = _randn((Hq, S, d), 21), _randn((Hkv, S, d), 22), _randn((Hkv, S, d), 23)
    qd, kd, vd = (rank_major(x, S, c, layout).to(dev()) for x in (q, k, v))
    o_run = torch.zeros((Hq, S, d), dtype=torch.float32, device=dev())
    l_run = torch.full((Hq, S), -float("inf"), dtype=torch.float32, device=dev())
    op = torch.empty_like(o_run)
    lp = torch.empty_like(l_run)
    for hop in range(c):
        for sub in range((S // c) // kvb):
            ra.fwd_hop_f32(qd, kd, vd, op, lp, c=c, causal=causal, layout=layout, kv_block=kvb, hop=hop, sub=sub)
            wo, wl = oring.ring_hop_partial(f64(q), f64(k), f64(v), c, layout, bool(causal), kvb, hop, sub)
            assert max_err(natural(op.cpu(), S, c, layout), wo) <= TOL_F32
            assert max_err(natural(lp.cpu(), S, c, layout), wl) <= TOL_F32
            ra.merge(o_run, l_run, op, lp)
    ro, rl = oatt.full_attention(f64(q), f64(k), f64(v), bool(causal))
    assert max_err(natural(o_run.cpu(), S, c, layout), ro) <= TOL_F32
    assert max_err(natural(l_run.cpu(), S, c, layout), rl) <= TOL_F32
    _status_ok(ra)


# ------------------------------------------------------------------ bf16 fused path

def _run_bf16(ra, q, k, v, c, layout, causal, kv_block):
    Hq, S, d = q.shape
    qd, kd, vd = (rank_major(x, S, c, layout).to(dev()) for x in (q, k, v))
    o = torch.full((Hq, S, d), float("nan"), dtype=torch.float32, device=dev())
    l = torch.full((Hq, S), float("nan"), dtype=torch.float32, device=dev())
    ra.fwd(qd, kd, vd, o, l, c=c, causal=causal, layout=layout, kv_block=kv_block)
    torch.cuda.synchronize()
    return natural(o.cpu(), S, c, layout), natural(l.cpu(), S, c, layout)


BF16_CASES = [
    # Hq, Hkv, S, d, c, layout, causal   (comment: pairing used by the kernel)
    (1, 1, 256, 64, 1, 0, 0),      # one head, tile pairs of positions
    (1, 1, 256, 64, 1, 0, 1),
    (2, 1, 256, 128, 1, 0, 1),     # head pairs
    (4, 2, 512, 64, 2, 1, 1),      # zigzag, chunk 128 -> head pairs
    (2, 2, 1024, 128, 4, 0, 1),    # chunk 256: position pairs
    (3, 3, 1024, 64, 2, 1, 1),     # zigzag chunk 256: position pairs
    (6, 2, 768, 64, 3, 0, 1),      # g = 3: single tiles
    (6, 2, 1536, 128, 3, 1, 1),    # g = 3 zigzag
    (2, 2, 512, 64, 4, 0, 1),      # chunk 128, one tile per chunk: single tiles
    (8, 1, 2048, 128, 2, 1, 0),    # g = 8 non-causal
    (4, 4, 640, 128, 5, 0, 1),     # c = 5, chunk 128
    (16, 2, 1024, 64, 4, 1, 1),    # g = 8 zigzag causal
]


@pytest.mark.parametrize("case", BF16_CASES)
def test_bf16_sweep(ra, case):
    Hq, Hkv, S, d, c, layout, causal = case
    m = S // (c * (2 if layout else 1))
    q = _randn((Hq, S, d), 31, torch.bfloat16)
    k = _randn((Hkv, S, d), 32, torch.bfloat16)
    v = _randn((Hkv, S, d), 33, torch.bfloat16)
    o, l = _run_bf16(ra, q, k, v, c, layout, causal, m)
    ro, rl = oatt.full_attention(f64(q), f64(k), f64(v), bool(causal))
    assert max_err(o, ro) <= TOL_BF16_OUT, max_err(o, ro)
    assert max_err(l, rl) <= TOL_BF16_LSE, max_err(l, rl)
    _status_ok(ra)


def test_bf16_causal_mha_4096_both_layouts(ra):
    """S=4096, 8 heads, d=64, c=4: contiguous (4 x 1024) and zigzag (8 x 512)."""
    from online_softmax_attention_zigzag_gb300.configs import CAUSAL_MHA_S4K as w, with_layout
    from online_softmax_attention_zigzag_gb300.inputs import make_qkv
    q, k, v = make_qkv(w)
    ro, rl = oatt.full_attention(f64(q), f64(k), f64(v), True)
    for layout in (0, 1):
        wl = with_layout(w, layout)
        o, l = _run_bf16(ra, q, k, v, wl.c, wl.layout, wl.causal, wl.kv_block)
        assert max_err(o, ro) <= TOL_BF16_OUT
        assert max_err(l, rl) <= TOL_BF16_LSE
    _status_ok(ra)


def test_bf16_natural_matches_rank_major(ra):
    """The chunk map folded into tile addressing gives bit-identical results."""
    Hq, Hkv, S, d, c = 8, 2, 2048, 128, 4
    q = _randn((Hq, S, d), 41, torch.bfloat16)
    k = _randn((Hkv, S, d), 42, torch.bfloat16)
    v = _randn((Hkv, S, d), 43, torch.bfloat16)
    for layout in (0, 1):
        o, l = _run_bf16(ra, q, k, v, c, layout, 1, 256)
        on = torch.empty((Hq, S, d), dtype=torch.float32, device=dev())
        ln = torch.empty((Hq, S), dtype=torch.float32, device=dev())
        ra.fwd_natural(q.to(dev()), k.to(dev()), v.to(dev()), on, ln, c=c, causal=1, layout=layout, kv_block=256)
        torch.cuda.synchronize()
        assert torch.equal(on.cpu(), o) and torch.equal(ln.cpu(), l)


@pytest.mark.parametrize("case", [
    # Hq, Hkv, S, d, c, layout, causal
    (8, 8, 4096, 64, 4, 0, 1),     # the 4096-token MHA workload, contiguous: position pairs
    (8, 8, 4096, 64, 4, 1, 1),     # and zigzag
    (6, 2, 1536, 128, 3, 1, 1),    # g = 3: single tiles
    (8, 2, 2048, 128, 4, 1, 0),    # head pairs, non-causal
])
def test_bf16_rank_restricted_matches_full(ra, case):
    """ringattn_fwd_rank writes exactly one rank's rows, bitwise equal to ringattn_fwd's."""
    Hq, Hkv, S, d, c, layout, causal = case
    n_r = S // c
    q = _randn((Hq, S, d), 61, torch.bfloat16)
    k = _randn((Hkv, S, d), 62, torch.bfloat16)
    v = _randn((Hkv, S, d), 63, torch.bfloat16)
    qd, kd, vd = (rank_major(x, S, c, layout).to(dev()) for x in (q, k, v))
    kvb = S // (c * (2 if layout else 1))
    of = torch.empty((Hq, S, d), dtype=torch.float32, device=dev())
    lf = torch.empty((Hq, S), dtype=torch.float32, device=dev())
    ra.fwd(qd, kd, vd, of, lf, c=c, causal=causal, layout=layout, kv_block=kvb)
    o = torch.full((Hq, S, d), float("nan"), dtype=torch.float32, device=dev())
    l = torch.full((Hq, S), float("nan"), dtype=torch.float32, device=dev())
    for r in range(c):
        ra.fwd_rank(qd, kd, vd, o, l, c=c, causal=causal, layout=layout, kv_block=kvb, rank=r)
        torch.cuda.synchronize()
        oc, lc = o.cpu(), l.cpu()
        done = slice(0, (r + 1) * n_r)
        assert torch.equal(oc[:, done], of.cpu()[:, done]) and torch.equal(lc[:, done], lf.cpu()[:, done])
        assert torch.isnan(oc[:, (r + 1) * n_r:]).all() and torch.isnan(lc[:, (r + 1) * n_r:]).all()
    ro, rl = oatt.full_attention(f64(q), f64(k), f64(v), bool(causal))
    assert max_err(natural(o.cpu(), S, c, layout), ro) <= TOL_BF16_OUT
    assert max_err(natural(l.cpu(), S, c, layout), rl) <= TOL_BF16_LSE
    _status_ok(ra)


@pytest.mark.parametrize("case", [(4, 2, 1024, 64, 2, 1, 1, 128), (2, 2, 1024, 128, 4, 0, 1, 128),
                                  (2, 1, 512, 64, 2, 0, 0, 256)])
def test_bf16_hop_partials_and_merge(ra, case):
    Hq, Hkv, S, d, c, layout, causal, kvb = case
    q = _randn((Hq, S, d), 51, torch.bfloat16)
    k = _randn((Hkv, S, d), 52, torch.bfloat16)
    v = _randn((Hkv, S, d), 53, torch.bfloat16)
    qd, kd, vd = (rank_major(x, S, c, layout).to(dev()) for x in (q, k, v))
    o_run = torch.zeros((Hq, S, d), dtype=torch.float32, device=dev())
    l_run = torch.full((Hq, S), -float("inf"), dtype=torch.float32, device=dev())
    op = torch.empty_like(o_run)
    lp = torch.empty_like(l_run)
    for hop in range(c):
        for sub in range((S // c) // kvb):
            ra.fwd_hop(qd, kd, vd, op, lp, c=c, causal=causal, layout=layout, kv_block=kvb, hop=hop, sub=sub)
            wo, wl = oring.ring_hop_partial(f64(q), f64(k), f64(v), c, layout, bool(causal), kvb, hop, sub)
            assert max_err(natural(op.cpu(), S, c, layout), wo) <= TOL_BF16_OUT
            assert max_err(natural(lp.cpu(), S, c, layout), wl) <= TOL_BF16_LSE
            ra.merge(o_run, l_run, op, lp)
    ro, rl = oatt.full_attention(f64(q), f64(k), f64(v), bool(causal))
    assert max_err(natural(o_run.cpu(), S, c, layout), ro) <= TOL_BF16_OUT
    assert max_err(natural(l_run.cpu(), S, c, layout), rl) <= TOL_BF16_LSE
    _status_ok(ra)


# ------------------------------------------------------------------ full-size workloads, sampled rows

def _sampled_check(ra, w, n_rows, fused=True, kv_block=None):
    from online_softmax_attention_zigzag_gb300.inputs import edge_rows, make_qkv, sample_rows
    q, k, v = make_qkv(w)
    out, lse = ra.attention(q.to(dev()), k.to(dev()), v.to(dev()), c=w.c, causal=w.causal, layout=w.layout,
                            kv_block=kv_block or w.kv_block)
    torch.cuda.synchronize()
    _status_ok(ra)
    errs = {}
    for name, (hs, ps) in (("sampled", sample_rows(w.bhq, w.seq, n_rows)),
                           ("edge", edge_rows(w.bhq, w.seq, w.n_chunks))):
        ro, rl = oatt.full_attention_rows(q, k, v, hs.numpy(), ps.numpy(), bool(w.causal))
        go = out[hs.to(dev()), ps.to(dev())].cpu()
        gl = lse[hs.to(dev()), ps.to(dev())].cpu()
        errs[name] = (max_err(go, ro), max_err(gl, rl))
    return errs, out, lse, (q, k, v)


def test_bf16_gqa_32k_sampled(ra):
    """S=32768, 64/8 heads, d=128, Q scaled by 1/sqrt(d), c=8 zigzag: 4096 rows + edge rows."""
    from online_softmax_attention_zigzag_gb300.configs import CAUSAL_GQA_S32K as w
    errs, *_ = _sampled_check(ra, w, 4096)
    for name, (eo, el) in errs.items():
        assert eo <= TOL_BF16_OUT and el <= TOL_BF16_LSE, (name, eo, el)


def test_bf16_gqa_128k_sampled(ra):
    """S=131072, 32/8 heads, d=128, c=16 zigzag: 4096 rows + edge rows."""
    from online_softmax_attention_zigzag_gb300.configs import CAUSAL_GQA_S128K as w
    errs, *_ = _sampled_check(ra, w, 4096)
    for name, (eo, el) in errs.items():
        assert eo <= TOL_BF16_OUT and el <= TOL_BF16_LSE, (name, eo, el)


@pytest.fixture(scope="module")
def outliers_64k(ra):
    """The non-causal B=2 S=65536 16-head workload (1% of Q/K entries x8, c=8 contiguous):
    rank-major device inputs, the fused result and the oracle on 4096 sampled rows plus
    the edge rows.  Shared by the fused check and the per-hop sweep."""
    from online_softmax_attention_zigzag_gb300.configs import NONCAUSAL_MHA_B2_S64K as w
    from online_softmax_attention_zigzag_gb300.inputs import edge_rows, make_qkv, sample_rows
    q, k, v = make_qkv(w)
    hs, ps = sample_rows(w.bhq, w.seq, 4096)
    he, pe = edge_rows(w.bhq, w.seq, w.n_chunks)
    hs, ps = torch.cat([hs, he]), torch.cat([ps, pe])
    ro, rl = oatt.full_attention_rows(q, k, v, hs.numpy(), ps.numpy(), False)
    qd, kd, vd = (torch.empty(x.shape, dtype=x.dtype, device=dev()) for x in (q, k, v))
    for src, dst in ((q, qd), (k, kd), (v, vd)):
        ra.permute(src.to(dev()), dst, c=w.c, layout=w.layout, inverse=0)
    del q, k, v
    o = torch.empty((w.bhq, w.seq, w.d), dtype=torch.float32, device=dev())
    l = torch.empty((w.bhq, w.seq), dtype=torch.float32, device=dev())
    ra.fwd(qd, kd, vd, o, l, c=w.c, causal=w.causal, layout=w.layout, kv_block=w.kv_block)
    on, ln = torch.empty_like(o), torch.empty_like(l)
    ra.permute(o, on, c=w.c, layout=w.layout, inverse=1)
    ra.permute(l, ln, c=w.c, layout=w.layout, inverse=1)
    torch.cuda.synchronize()
    _status_ok(ra)
    del o, l
    yield dict(w=w, qkv=(qd, kd, vd), rows=(hs, ps), oracle=(ro, rl), fused=(on, ln))
    torch.cuda.empty_cache()


def test_bf16_noncausal_outliers_64k_fused(ra, outliers_64k):
    """Fused path on 4096 sampled rows and the edge rows against the oracle."""
    hs, ps = outliers_64k["rows"]
    ro, rl = outliers_64k["oracle"]
    on, ln = outliers_64k["fused"]
    hd, pd = hs.to(dev()), ps.to(dev())
    assert max_err(on[hd, pd].cpu(), ro) <= TOL_BF16_OUT
    assert max_err(ln[hd, pd].cpu(), rl) <= TOL_BF16_LSE


@pytest.mark.parametrize("kv_block", [512, 1024, 2048, 4096, 8192])
def test_bf16_noncausal_outliers_64k_per_hop_sweep(ra, outliers_64k, kv_block):
    """The ring-faithful per-hop path at every message size of the sweep: one
    ringattn_fwd_hop partial per message (c hops x chunk / kv_block sub-blocks), each
    folded into the running result by the merge kernel.  The folded result against the
    oracle on the sampled and edge rows, and against the fused result everywhere."""
    w = outliers_64k["w"]
    qd, kd, vd = outliers_64k["qkv"]
    hs, ps = outliers_64k["rows"]
    ro, rl = outliers_64k["oracle"]
    on, ln = outliers_64k["fused"]
    S, c = w.seq, w.c
    o_run = torch.zeros((w.bhq, S, w.d), dtype=torch.float32, device=dev())
    l_run = torch.full((w.bhq, S), -float("inf"), dtype=torch.float32, device=dev())
    op, lp = torch.empty_like(o_run), torch.empty_like(l_run)
    for hop in range(c):
        for sub in range((S // c) // kv_block):
            ra.fwd_hop(qd, kd, vd, op, lp, c=c, causal=w.causal, layout=w.layout, kv_block=kv_block, hop=hop,
                       sub=sub)
            ra.merge(o_run, l_run, op, lp)
    del op, lp
    o_nat, l_nat = torch.empty_like(o_run), torch.empty_like(l_run)
    ra.permute(o_run, o_nat, c=c, layout=w.layout, inverse=1)
    ra.permute(l_run, l_nat, c=c, layout=w.layout, inverse=1)
    torch.cuda.synchronize()
    _status_ok(ra)
    del o_run, l_run
    hd, pd = hs.to(dev()), ps.to(dev())
    assert max_err(o_nat[hd, pd].cpu(), ro) <= TOL_BF16_OUT
    assert max_err(l_nat[hd, pd].cpu(), rl) <= TOL_BF16_LSE
    assert (o_nat - on).abs().max().item() <= TOL_BF16_OUT
    assert (l_nat - ln).abs().max().item() <= TOL_BF16_LSE


# ------------------------------------------------------------------ failure path

def test_bounded_wait_gives_up_and_context_survives(ra):
    ra.selftest_timeout(5_000_000)  # 5 ms
    assert ra.sync_status() == ra.RA_ERR_TIMEOUT
    assert ra.sync_status() == ra.RA_OK  # the record was cleared
    # the context is still usable
    q = _randn((2, 256, 64), 61, torch.bfloat16)
    o, l = _run_bf16(ra, q, q[:1].contiguous(), q[:1].contiguous(), 1, 0, 1, 256)
    ro, rl = oatt.full_attention(f64(q), f64(q[:1]), f64(q[:1]), True)
    assert max_err(o, ro) <= TOL_BF16_OUT
    _status_ok(ra)


def test_binding_raises_on_bad_arguments(ra):
    q = torch.zeros((2, 4000, 64), dtype=torch.bfloat16, device=dev())
    o = torch.zeros((2, 4000, 64), dtype=torch.float32, device=dev())
    l = torch.zeros((2, 4000), dtype=torch.float32, device=dev())
    with pytest.raises(ra.RingAttnError) as e:
        ra.fwd(q, q, q, o, l, c=3, causal=1, layout=1, kv_block=128)
    assert e.value.code == ra.RA_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        ra.fwd(q.float(), q, q, o, l, c=4, causal=1, layout=1, kv_block=128)
