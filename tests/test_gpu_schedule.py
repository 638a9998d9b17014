"""Dynamic work-item draw of the fused kernels: every launch takes a pair of counters from a
ring of 256 slots in device memory and its last CTA zeroes them again.  Many launches in
a row (more than the ring holds, forward and backward interleaved, two streams) must give
bitwise the same results as the first, and agree with the oracle."""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from tests.gpu_util import TOL_BF16_LSE, TOL_BF16_OUT, dev, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    from online_softmax_attention_zigzag_gb300 import ringattn
    ringattn.lib()
    torch.cuda.set_device(0)
    return ringattn


def _randn(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float32) * scale).to(torch.bfloat16)


def test_counter_slots_wrap_forward_and_backward(ra):
    Hq, Hkv, S, d, c = 4, 2, 1024, 128, 4
    kw = dict(c=c, causal=1, layout=1, kv_block=S // (2 * c))
    q = _randn((Hq, S, d), 301, d ** -0.5).to(dev())
    k, v = _randn((Hkv, S, d), 302).to(dev()), _randn((Hkv, S, d), 303).to(dev())
    dout = _randn((Hq, S, d), 304).to(dev())
    out = torch.empty((Hq, S, d), dtype=torch.float32, device=dev())
    lse = torch.empty((Hq, S), dtype=torch.float32, device=dev())
    grads = [torch.empty((Hq, S, d), dtype=torch.float32, device=dev()),
             torch.empty((Hkv, S, d), dtype=torch.float32, device=dev()),
             torch.empty((Hkv, S, d), dtype=torch.float32, device=dev())]
    delta = torch.empty((Hq, S), dtype=torch.float32, device=dev())
    ra.fwd_natural(q, k, v, out, lse, **kw)
    ra.bwd(q, k, v, out, lse, dout, *grads, delta, natural=True, **kw)
    torch.cuda.synchronize()
    assert ra.sync_status() == ra.RA_OK
    ref = [out.clone(), lse.clone()] + [g.clone() for g in grads]
    side = torch.cuda.Stream()
    o2, l2 = torch.empty_like(out), torch.empty_like(lse)
    for i in range(200):  # 200 forwards + 2 x 100 backward launches: past the 256 slots
        ra.fwd_natural(q, k, v, out, lse, **kw)
        with torch.cuda.stream(side):  # a second stream drawing slots at the same time
            ra.fwd_natural(q, k, v, o2, l2, stream=side.cuda_stream, **kw)
        if i % 2 == 0:
            ra.bwd(q, k, v, ref[0], ref[1], dout, *grads, delta, natural=True, **kw)
    torch.cuda.synchronize()
    assert ra.sync_status() == ra.RA_OK
    for got, want in zip([out, lse, o2, l2] + grads, ref[:2] + ref[:2] + ref[2:]):
        assert torch.equal(got, want)
    ro, rl = oatt.full_attention(f64(q.cpu()), f64(k.cpu()), f64(v.cpu()), True)
    assert np.abs(out.cpu().double().numpy() - ro).max() <= TOL_BF16_OUT
    assert np.abs(lse.cpu().double().numpy() - rl).max() <= TOL_BF16_LSE
