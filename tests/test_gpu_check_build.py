"""The check build (libringattn_check.so, compiled with -DRA_CHECK) against the normal library.

The check build puts an index check at every place a kernel derives a memory index from
the chunk and work-item arithmetic; a failed check records RA_ERR_BOUNDS instead of
touching memory outside the tensor.  On valid inputs no check may fail and the results
must be bitwise those of the normal library.  Outputs start as NaN, so a row that a
kernel never writes shows up as NaN.

Both libraries are loaded into this process through two instances of the binding; each
has its own device error word, read by its own ringattn_sync_status.
"""
import importlib.util
import os

import numpy as np
import pytest
import torch

from tests.gpu_util import dev, rank_major

pytestmark = pytest.mark.gpu

PKG = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "online_softmax_attention_zigzag_gb300")


def _binding(lib_name, module_name):
    spec = importlib.util.spec_from_file_location(module_name, os.path.join(PKG, "ringattn.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.LIB_PATH = os.path.join(PKG, lib_name)
    mod.lib()
    return mod


@pytest.fixture(scope="module")
def libs():
    torch.cuda.set_device(0)
    return _binding("libringattn.so", "ringattn_release"), _binding("libringattn_check.so", "ringattn_checked")


def _randn(shape, seed, dtype=torch.bfloat16, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(dtype)


def _nan(shape):
    return torch.full(shape, float("nan"), dtype=torch.float32, device=dev())


def _both(libs, run):
    """run(ra) -> tuple of output tensors; returns the release and check results after
    confirming that neither library recorded an error."""
    res = []
    for ra in libs:
        out = run(ra)
        torch.cuda.synchronize()
        assert ra.sync_status() == ra.RA_OK, ra.__name__
        res.append(tuple(t.cpu() for t in out))
    return res


def _same(a, b):
    for x, y in zip(a, b):
        assert not torch.isnan(x).any(), "a row was never written"
        assert torch.equal(x, y)


@pytest.mark.parametrize("case", [
    # Hq, Hkv, S, d, c, layout, causal
    (4, 2, 512, 64, 2, 1, 1),      # head pairs, zigzag
    (2, 2, 1024, 128, 4, 0, 1),    # position pairs, contiguous
    (6, 2, 768, 64, 3, 0, 1),      # single tiles
    (8, 1, 1024, 128, 2, 1, 0),    # non-causal
])
def test_forward_entry_points(libs, case):
    Hq, Hkv, S, d, c, layout, causal = case
    m = S // (c * (2 if layout else 1))
    q, k, v = _randn((Hq, S, d), 1), _randn((Hkv, S, d), 2), _randn((Hkv, S, d), 3)
    qd, kd, vd = (rank_major(x, S, c, layout).to(dev()) for x in (q, k, v))
    qn, kn, vn = q.to(dev()), k.to(dev()), v.to(dev())
    kw = dict(c=c, causal=causal, layout=layout, kv_block=m)

    def fused(ra):
        o, l = _nan((Hq, S, d)), _nan((Hq, S))
        ra.fwd(qd, kd, vd, o, l, **kw)
        on, ln = _nan((Hq, S, d)), _nan((Hq, S))
        ra.fwd_natural(qn, kn, vn, on, ln, **kw)
        orr, lr = _nan((Hq, S, d)), _nan((Hq, S))
        for r in range(c):
            ra.fwd_rank(qd, kd, vd, orr, lr, rank=r, **kw)
        return o, l, on, ln, orr, lr

    _same(*_both(libs, fused))

    def per_hop(ra):
        o, l = torch.zeros((Hq, S, d), dtype=torch.float32, device=dev()), _nan((Hq, S))
        l.fill_(-float("inf"))
        op, lp = _nan((Hq, S, d)), _nan((Hq, S))
        for hop in range(c):
            ra.fwd_hop(qd, kd, vd, op, lp, hop=hop, sub=0, **kw)
            ra.merge(o, l, op, lp)
        return o, l

    _same(*_both(libs, per_hop))


def test_permute_and_fp32_path(libs):
    S, H, c = 96, 3, 3
    g = torch.Generator().manual_seed(4)
    x = torch.randint(0, 256, (H, S, 6), generator=g, dtype=torch.uint8).to(dev())

    def permute(ra):
        y, z = torch.empty_like(x), torch.empty_like(x)
        ra.permute(x, y, c=c, layout=1, inverse=0)
        ra.permute(y, z, c=c, layout=1, inverse=1)
        return y, z

    (y0, z0), (y1, z1) = _both(libs, permute)
    assert torch.equal(y0, y1) and torch.equal(z0, z1) and torch.equal(z1, x.cpu())
    q, k, v = (_randn((2, 48, 8), s, torch.float32).to(dev()) for s in (5, 6, 7))

    def f32(ra):
        o, l = _nan((2, 48, 8)), _nan((2, 48))
        ra.fwd_f32(q, k, v, o, l, c=3, causal=1, layout=1, kv_block=8)
        return o, l

    _same(*_both(libs, f32))


def test_docmask_and_backward(libs):
    Hq, Hkv, S, d, c, layout = 4, 2, 1024, 128, 2, 1
    lens = [100, 1, 400, 23, 500]
    doc = torch.repeat_interleave(torch.arange(len(lens), dtype=torch.int32), torch.tensor(lens)).to(dev())
    q, k, v = _randn((Hq, S, d), 11, scale=0.1), _randn((Hkv, S, d), 12), _randn((Hkv, S, d), 13)
    dout = _randn((Hq, S, d), 14)
    qd, kd, vd, dod = (rank_major(x, S, c, layout).to(dev()) for x in (q, k, v, dout))

    def docmask(ra):
        o, l, ds = _nan((Hq, S, d)), _nan((Hq, S)), torch.empty((S,), dtype=torch.int32, device=dev())
        ra.fwd_docmask(qd, kd, vd, o, l, doc, ds, c=c, layout=layout)
        o2, l2 = _nan((Hq, S, d)), _nan((Hq, S))
        ra.fwd_docmask_noalloc(qd, kd, vd, o2, l2, doc, c=c, layout=layout)
        return o, l, o2, l2

    _same(*_both(libs, docmask))
    kw = dict(c=c, causal=1, layout=layout, kv_block=S // (2 * c))

    def backward(ra):
        o, l = _nan((Hq, S, d)), _nan((Hq, S))
        ra.fwd(qd, kd, vd, o, l, **kw)
        dq, dk, dv = _nan((Hq, S, d)), _nan((Hkv, S, d)), _nan((Hkv, S, d))
        delta = _nan((Hq, S))
        ra.bwd(qd, kd, vd, o, l, dod, dq, dk, dv, delta, **kw)
        return dq, dk, dv

    _same(*_both(libs, backward))


def test_ulysses(libs):
    Hq, Hkv, S, d, c, layout = 8, 2, 1024, 64, 4, 1
    q, k, v = _randn((Hq, S, d), 21), _randn((Hkv, S, d), 22), _randn((Hkv, S, d), 23)
    order = torch.from_numpy(np.concatenate([
        np.concatenate([np.arange(ch * (S // 8), (ch + 1) * (S // 8)) for ch in (r, 2 * c - 1 - r)])
        for r in range(c)]))
    seq = [x[:, order].transpose(0, 1).contiguous().to(dev()) for x in (q, k, v)]   # [S, H, d]

    def uly(ra):
        o, l = _nan((S, Hq, d)), _nan((S, Hq))
        ws = torch.empty(ra.host_workspace_bytes(S, Hq, Hkv, d), dtype=torch.uint8, device=dev())
        ra.ulysses_fwd(*seq, o, l, ws, c=c, causal=1, layout=layout)
        return o, l

    _same(*_both(libs, uly))
