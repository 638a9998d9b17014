"""The fused kernel writes `out` with 32-byte stores when `out` is 32-byte aligned and with
16-byte stores otherwise (the ABI requires 16).  Both paths give bitwise the same result."""
import pytest
import torch

from tests.gpu_util import dev

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


@pytest.mark.parametrize("d", [64, 128])
def test_out_16_byte_aligned_equals_32_byte_aligned(ra, d):
    Hq, Hkv, S, c = 4, 2, 1024, 2
    kw = dict(c=c, causal=1, layout=1, kv_block=S // (2 * c))
    q = _randn((Hq, S, d), 401, d ** -0.5).to(dev())
    k, v = _randn((Hkv, S, d), 402).to(dev()), _randn((Hkv, S, d), 403).to(dev())
    n = Hq * S * d
    buf = torch.full((n + 8,), float("nan"), dtype=torch.float32, device=dev())
    out_a = buf[:n].view(Hq, S, d)          # 256-byte aligned (allocator)
    lse = torch.empty((Hq, S), dtype=torch.float32, device=dev())
    ra.fwd_natural(q, k, v, out_a, lse, **kw)
    want = out_a.clone()
    buf.fill_(float("nan"))
    out_u = buf[4:4 + n].view(Hq, S, d)     # 16 bytes past a 32-byte boundary
    assert out_u.data_ptr() % 32 == 16
    ra.fwd_natural(q, k, v, out_u, lse, **kw)
    torch.cuda.synchronize()
    assert ra.sync_status() == ra.RA_OK
    assert torch.equal(out_u, want)
    assert torch.isnan(buf[:4]).all() and torch.isnan(buf[4 + n:]).all()  # nothing written outside
