"""Masked scores far above the visible ones, on the GPU against the oracle.

The fused kernel takes a tile's row max from its TMEM loads when no score of the warp is
masked, and computes it after masking otherwise.  These inputs make masked scores far
larger than every visible one (future keys on the causal diagonal, up to 127 above; keys
of an earlier document under the document mask, 400 above): a max taken over masked scores
would push the visible exp2 values below fp32's range for many rows (302 of 1024 in the
first causal case), which would come out empty, far outside the bf16 tolerances.  ("Ring Attention and Ulysses shard a sequence two different ways",
the online-softmax update: the running max is over the keys a row may see.)
"""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import docmask as odoc
from tests.gpu_util import TOL_BF16_LSE, TOL_BF16_OUT, dev, f64, max_err, natural, rank_major

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    from online_softmax_attention_zigzag_gb300 import ringattn
    ringattn.lib()
    return ringattn


def _small(shape, seed, scale):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32) * scale


def _rising_scores(Hq, Hkv, S, d, seed):
    """q_i . k_j = j - i plus small noise (two features: q_i = (1, -i), k_j = (j, 1), as bf16
    rounds them): every key a row may see scores at most ~0, every later key more, up to 127
    above on the row's diagonal tile, so a max over those would flush the row's exp2 to
    zero; the scores stay small enough for fp32 to hold lse well inside 1e-3."""
    q = _small((Hq, S, d), seed, 0.05)
    k = _small((Hkv, S, d), seed + 1, 0.05)
    pos = torch.arange(S, dtype=torch.float32)
    q[:, :, 0] = 1.0
    q[:, :, 1] = -pos
    k[:, :, 0] = pos
    k[:, :, 1] = 1.0
    v = _small((Hkv, S, d), seed + 2, 1.0)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


@pytest.mark.parametrize("Hq,Hkv,S,d,c,layout", [
    (2, 1, 1024, 128, 2, 1),
    (4, 2, 768, 64, 3, 0),
])
def test_causal_diagonal_with_high_future_scores(ra, Hq, Hkv, S, d, c, layout):
    q, k, v = _rising_scores(Hq, Hkv, S, d, 301)
    qd, kd, vd = (rank_major(x, S, c, layout).to(dev()) for x in (q, k, v))
    o = torch.full((Hq, S, d), float("nan"), dtype=torch.float32, device=dev())
    l = torch.full((Hq, S), float("nan"), dtype=torch.float32, device=dev())
    m = S // (c * (2 if layout else 1))
    ra.fwd(qd, kd, vd, o, l, c=c, causal=1, layout=layout, kv_block=m)
    assert ra.sync_status() == ra.RA_OK
    o, l = natural(o.cpu(), S, c, layout), natural(l.cpu(), S, c, layout)
    ro, rl = oatt.full_attention(f64(q), f64(k), f64(v), True)
    assert np.isfinite(o.numpy()).all() and np.isfinite(l.numpy()).all()
    assert max_err(o, ro) <= TOL_BF16_OUT, max_err(o, ro)
    assert max_err(l, rl) <= TOL_BF16_LSE, max_err(l, rl)


@pytest.mark.parametrize("d,lens", [
    (128, [200, 300, 524]),
    (64, [64, 1, 191, 256, 500, 12]),
])
def test_docmask_with_high_scores_in_earlier_documents(ra, d, lens):
    """Keys of even-numbered documents score 400 against every query, keys of odd ones ~0:
    a row of an odd document shares key tiles with the preceding even document's keys,
    which it may not see."""
    Hq, Hkv, c, layout = 2, 1, 2, 1
    doc = torch.repeat_interleave(torch.arange(len(lens), dtype=torch.int32), torch.tensor(lens))
    S = len(doc)
    q = _small((Hq, S, d), 311, 0.05)
    k = _small((Hkv, S, d), 312, 0.05)
    q[:, :, 0] = 1.0
    k[:, :, 0] = torch.where(doc % 2 == 0, 400.0, 0.0)
    v = _small((Hkv, S, d), 313, 1.0)
    q, k, v = (x.to(torch.bfloat16) for x in (q, k, v))
    qd, kd, vd = (rank_major(x, S, c, layout).to(dev()) for x in (q, k, v))
    o = torch.full((Hq, S, d), float("nan"), dtype=torch.float32, device=dev())
    l = torch.full((Hq, S), float("nan"), dtype=torch.float32, device=dev())
    ds = torch.empty((S,), dtype=torch.int32, device=dev())
    ra.fwd_docmask(qd, kd, vd, o, l, doc.to(dev()), ds, c=c, layout=layout)
    assert ra.sync_status() == ra.RA_OK
    o, l = natural(o.cpu(), S, c, layout), natural(l.cpu(), S, c, layout)
    ro, rl = odoc.doc_attention(f64(q), f64(k), f64(v), doc.numpy())
    assert np.isfinite(o.numpy()).all() and np.isfinite(l.numpy()).all()
    assert max_err(o, ro) <= TOL_BF16_OUT, max_err(o, ro)
    assert max_err(l, rl) <= TOL_BF16_LSE, max_err(l, rl)
