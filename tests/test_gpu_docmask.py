"""Document-masked attention over all-gathered K/V on the GPU against the oracle
(ringattn_fwd_docmask; "Interrogating parallelism, part 5", "Why did Llama 3 not use a
ring?").  Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

from oracle import docmask as odoc
from tests.gpu_util import TOL_BF16_LSE, TOL_BF16_OUT, dev, f64, max_err, natural, rank_major

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    from online_softmax_attention_zigzag_gb300 import ringattn
    ringattn.lib()
    return ringattn


def _randn(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _run(ra, q, k, v, doc, c, layout):
    Hq, S, d = q.shape
    qd, kd, vd = (rank_major(x, S, c, layout).to(dev()) for x in (q, k, v))
    o = torch.full((Hq, S, d), float("nan"), dtype=torch.float32, device=dev())
    l = torch.full((Hq, S), float("nan"), dtype=torch.float32, device=dev())
    ds = torch.full((S,), -7, dtype=torch.int32, device=dev())
    ra.fwd_docmask(qd, kd, vd, o, l, doc.to(torch.int32).to(dev()), ds, c=c, layout=layout)
    assert ra.sync_status() == ra.RA_OK
    return natural(o.cpu(), S, c, layout), natural(l.cpu(), S, c, layout), ds.cpu()


def _doc_from_lengths(lens):
    return torch.repeat_interleave(torch.arange(len(lens), dtype=torch.int32), torch.tensor(lens))


CASES = [
    # Hq, Hkv, d, c, layout, document lengths (sum = S)
    (2, 2, 64, 1, 0, [256]),                                 # one document: plain causal attention
    (4, 2, 128, 2, 1, [1, 127, 128, 1, 1, 254]),              # boundaries on and off tile edges
    (8, 2, 128, 4, 1, [300, 5, 700, 1, 18]),                  # GQA head pairs, zigzag
    (3, 3, 64, 2, 0, [100, 404, 1, 1, 6]),                    # MHA position pairs, contiguous
    (6, 2, 128, 3, 1, [768]),                                 # g = 3: single tiles
    (2, 1, 64, 2, 1, [1] * 512),                              # every token its own document
]


@pytest.mark.parametrize("case", CASES)
def test_docmask_vs_oracle(ra, case):
    Hq, Hkv, d, c, layout, lens = case
    doc = _doc_from_lengths(lens)
    S = len(doc)
    q, k, v = _randn((Hq, S, d), 81), _randn((Hkv, S, d), 82), _randn((Hkv, S, d), 83)
    o, l, ds = _run(ra, q, k, v, doc, c, layout)
    ro, rl = odoc.doc_attention(f64(q), f64(k), f64(v), doc.numpy())
    assert max_err(o, ro) <= TOL_BF16_OUT, max_err(o, ro)
    assert max_err(l, rl) <= TOL_BF16_LSE, max_err(l, rl)
    # the scratch holds every position's document start, bit-exact
    d_np = doc.numpy()
    assert np.array_equal(ds.numpy(), np.searchsorted(d_np, d_np, side="left"))


def test_docmask_single_token_documents_give_v(ra):
    """A document of one token sees only itself: out is v_i exactly (P = 1 in bf16)."""
    Hq, Hkv, S, d = 2, 2, 512, 128
    q, k, v = _randn((Hq, S, d), 84), _randn((Hkv, S, d), 85), _randn((Hkv, S, d), 86)
    o, l, _ = _run(ra, q, k, v, torch.arange(S, dtype=torch.int32), 2, 1)
    assert torch.equal(o, v.to(torch.float32))
    ql = (f64(q) * f64(k)).sum(-1)
    assert max_err(l, ql) <= TOL_BF16_LSE


def test_docmask_one_document_matches_causal_ring(ra):
    """With a single document the mask is the causal mask: agrees with ringattn_fwd."""
    Hq, Hkv, S, d, c = 8, 2, 2048, 128, 4
    q, k, v = _randn((Hq, S, d), 87), _randn((Hkv, S, d), 88), _randn((Hkv, S, d), 89)
    o, l, _ = _run(ra, q, k, v, torch.zeros(S, dtype=torch.int32), c, 1)
    qd, kd, vd = (rank_major(x, S, c, 1).to(dev()) for x in (q, k, v))
    oc = torch.empty((Hq, S, d), dtype=torch.float32, device=dev())
    lc = torch.empty((Hq, S), dtype=torch.float32, device=dev())
    ra.fwd(qd, kd, vd, oc, lc, c=c, causal=1, layout=1, kv_block=S // (2 * c))
    torch.cuda.synchronize()
    # the two kernels visit the keys in different orders (natural vs ring): rounding only
    assert max_err(o, natural(oc.cpu(), S, c, 1)) <= TOL_BF16_OUT
    assert max_err(l, natural(lc.cpu(), S, c, 1)) <= TOL_BF16_LSE


def test_docmask_4096_workload_all_rows(ra):
    """S=4096, 8/2 heads, d=128, c=4 zigzag, documents of 1..2048 tokens: every row."""
    from online_softmax_attention_zigzag_gb300.configs import DOCMASK_GQA_S4K as w
    from online_softmax_attention_zigzag_gb300.inputs import doc_ids, make_qkv
    q, k, v = make_qkv(w)
    doc = doc_ids(w.seq, *w.doc_len)
    o, l, _ = _run(ra, q, k, v, doc, w.c, w.layout)
    ro, rl = odoc.doc_attention(f64(q), f64(k), f64(v), doc.numpy())
    assert max_err(o, ro) <= TOL_BF16_OUT and max_err(l, rl) <= TOL_BF16_LSE


def test_docmask_32k_sampled_and_document_edges(ra):
    """S=32768, 64/8 heads, d=128, c=8 zigzag, documents of 32..8192 tokens: 2048 sampled
    rows plus the first and last token of every document in heads 0 and 63."""
    from online_softmax_attention_zigzag_gb300.configs import DOCMASK_GQA_S32K as w
    from online_softmax_attention_zigzag_gb300.inputs import doc_ids, make_qkv, sample_rows
    q, k, v = make_qkv(w)
    doc = doc_ids(w.seq, *w.doc_len)
    qd, kd, vd = (torch.empty(x.shape, dtype=x.dtype, device=dev()) for x in (q, k, v))
    for src, dst in ((q, qd), (k, kd), (v, vd)):
        ra.permute(src.to(dev()), dst, c=w.c, layout=w.layout, inverse=0)
    o = torch.empty((w.bhq, w.seq, w.d), dtype=torch.float32, device=dev())
    l = torch.empty((w.bhq, w.seq), dtype=torch.float32, device=dev())
    ds = torch.empty((w.seq,), dtype=torch.int32, device=dev())
    ra.fwd_docmask(qd, kd, vd, o, l, doc.to(dev()), ds, c=w.c, layout=w.layout)
    on, ln = torch.empty_like(o), torch.empty_like(l)
    ra.permute(o, on, c=w.c, layout=w.layout, inverse=1)
    ra.permute(l, ln, c=w.c, layout=w.layout, inverse=1)
    assert ra.sync_status() == ra.RA_OK
    d_np = doc.numpy()
    starts = np.nonzero(np.r_[True, d_np[1:] != d_np[:-1]])[0]
    ends = np.r_[starts[1:] - 1, w.seq - 1]
    edge_pos = np.unique(np.r_[starts, ends])
    hs_e = np.repeat([0, w.bhq - 1], len(edge_pos))
    ps_e = np.tile(edge_pos, 2)
    hs, ps = sample_rows(w.bhq, w.seq, 2048)
    for name, (h, p) in (("sampled", (hs.numpy(), ps.numpy())), ("edges", (hs_e, ps_e))):
        ro, rl = odoc.doc_attention_rows(q, k, v, doc, h, p)
        hh, pp = torch.from_numpy(h).to(dev()), torch.from_numpy(p).to(dev())
        eo = max_err(on[hh, pp].cpu(), ro)
        el = max_err(ln[hh, pp].cpu(), rl)
        assert eo <= TOL_BF16_OUT and el <= TOL_BF16_LSE, (name, eo, el)
