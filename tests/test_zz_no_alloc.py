"""ringattn_fwd_docmask_noalloc against ringattn_fwd_docmask, through the C ABI.

The no-allocation entry point serves callers that cannot call cudaMalloc where they run
attention (a fixed memory budget handed out up front, a plug-in whose host owns every
allocation, code that must avoid the synchronisation an allocation can cause): they pass
no scratch, and the document starts go to a static device array inside the library.  Its
result must be that of the entry point with caller-owned scratch.

Both entry points run the same two kernels on the same inputs, so the results must be
bitwise equal: a partly stale scratch would change some rows and show here.  Two calls in
a row with different packings and lengths check that what the first call leaves in the
shared array does not leak into the second, and sampled rows of each call are checked
against the float64 oracle (document-masked attention), so the result is right on its own
and not only equal to the other entry point's.  This file is named to be collected last,
so a run that stops at the first failure has run every other test first.
"""
import ctypes

import pytest
import torch

from oracle import docmask as odoc
from tests.gpu_util import TOL_BF16_LSE, TOL_BF16_OUT, dev, max_err, natural, rank_major

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    from online_softmax_attention_zigzag_gb300 import ringattn
    ringattn.lib()
    return ringattn


def _randn(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _doc(lens):
    return torch.repeat_interleave(torch.arange(len(lens), dtype=torch.int32), torch.tensor(lens))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _both(ra, Hq, Hkv, d, c, layout, lens, seed):
    """Run both entry points on the same inputs, on the current stream; return
    (out, lse) of the no-allocation call and of the caller-scratch call."""
    doc = _doc(lens)
    S = len(doc)
    q, k, v = _randn((Hq, S, d), seed), _randn((Hkv, S, d), seed + 1), _randn((Hkv, S, d), seed + 2)
    qd, kd, vd = (rank_major(x, S, c, layout).to(dev()) for x in (q, k, v))
    ids = doc.to(dev())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    res = []
    for noalloc in (True, False):
        o = torch.full((Hq, S, d), float("nan"), dtype=torch.float32, device=dev())
        l = torch.full((Hq, S), float("nan"), dtype=torch.float32, device=dev())
        if noalloc:
            st = ra.lib().ringattn_fwd_docmask_noalloc(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(o), _ptr(l), _ptr(ids),
                                                      S, Hq, Hkv, d, c, layout, stream)
        else:
            scratch = torch.empty((S,), dtype=torch.int32, device=dev())
            st = ra.lib().ringattn_fwd_docmask(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(o), _ptr(l), _ptr(ids),
                                               _ptr(scratch), S, Hq, Hkv, d, c, layout, stream)
        assert st == ra.RA_OK, ra.strerror(st)
        res.append((o, l))
    assert ra.sync_status() == ra.RA_OK
    # sampled rows of the no-allocation result against the oracle (natural order)
    g = torch.Generator().manual_seed(seed + 3)
    starts = torch.cumsum(torch.tensor([0] + list(lens[:-1])), 0)        # every document's first row
    ps = torch.cat([torch.randint(0, S, (88,), generator=g), starts, torch.tensor([S - 1])])
    hs = torch.randint(0, Hq, (len(ps),), generator=g)
    on, ln = natural(res[0][0].cpu(), S, c, layout), natural(res[0][1].cpu(), S, c, layout)
    ro, rl = odoc.doc_attention_rows(q, k, v, doc.numpy(), hs.numpy(), ps.numpy())
    assert max_err(on[hs, ps], ro) <= TOL_BF16_OUT, max_err(on[hs, ps], ro)
    assert max_err(ln[hs, ps], rl) <= TOL_BF16_LSE, max_err(ln[hs, ps], rl)
    return [(o.cpu(), l.cpu()) for o, l in res]


def test_noalloc_matches_caller_scratch_on_two_calls_in_a_row(ra):
    # first call: 4096 positions, long and short documents, GQA head pairs, zigzag
    (o1, l1), (r1, s1) = _both(ra, 8, 2, 128, 4, 1, [1, 900, 127, 2000, 3, 1065], 301)
    # second call: shorter sequence and other boundaries, MHA position pairs, contiguous;
    # the static array still holds the first call's 4096 document starts
    (o2, l2), (r2, s2) = _both(ra, 3, 3, 64, 2, 0, [300, 1, 500, 1, 222], 311)
    for o, l, r, s in ((o1, l1, r1, s1), (o2, l2, r2, s2)):
        assert torch.isfinite(o).all() and torch.isfinite(l).all()
        assert torch.equal(o, r) and torch.equal(l, s)


def test_noalloc_rejects_sequences_beyond_its_scratch(ra):
    S = ra.DOCMASK_NOALLOC_MAX_S + 256
    buf = torch.empty((16,), dtype=torch.int32, device=dev())
    p = _ptr(buf)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = ra.lib().ringattn_fwd_docmask_noalloc(p, p, p, p, p, p, S, 1, 1, 64, 1, 0, stream)
    assert st == ra.RA_ERR_UNSUPPORTED
