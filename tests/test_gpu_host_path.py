"""ringattn_fwd_host (host buffers in and out, copies overlapped with the attention by
KV-head groups) against the oracle and against ringattn_fwd_natural on device buffers.
Every call goes through the C ABI."""
import pytest
import torch

from oracle import attention as oatt
from tests.gpu_util import TOL_BF16_LSE, TOL_BF16_OUT, dev, f64, max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    from online_softmax_attention_zigzag_gb300 import ringattn
    ringattn.lib()
    torch.cuda.set_device(0)
    return ringattn


def _randn(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _host_call(ra, q, k, v, kw, pin=True):
    Hq, S, d = q.shape
    if pin:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    out = torch.full((Hq, S, d), float("nan"), dtype=torch.float32, pin_memory=pin)
    lse = torch.full((Hq, S), float("nan"), dtype=torch.float32, pin_memory=pin)
    ws = torch.empty(ra.host_workspace_bytes(S, Hq, k.shape[0], d), dtype=torch.uint8, device=dev())
    ra.fwd_host(q, k, v, out, lse, ws, **kw)
    assert ra.sync_status() == ra.RA_OK
    return out, lse


def _device_call(ra, q, k, v, kw):
    Hq, S, d = q.shape
    o = torch.empty((Hq, S, d), dtype=torch.float32, device=dev())
    l = torch.empty((Hq, S), dtype=torch.float32, device=dev())
    ra.fwd_natural(q.to(dev()), k.to(dev()), v.to(dev()), o, l, **kw)
    assert ra.sync_status() == ra.RA_OK
    return o.cpu(), l.cpu()


@pytest.mark.parametrize("pin", [True, False])
def test_host_path_small_vs_oracle(ra, pin):
    """S=2048, 8/2 heads, d=128, c=4 zigzag causal: one group; every row against the oracle,
    and bitwise against the device-buffer call.  Pageable buffers give the same result."""
    Hq, Hkv, S, d = 8, 2, 2048, 128
    q, k, v = _randn((Hq, S, d), 51), _randn((Hkv, S, d), 52), _randn((Hkv, S, d), 53)
    kw = dict(c=4, causal=1, layout=1, kv_block=256)
    out, lse = _host_call(ra, q, k, v, kw, pin=pin)
    ro, rl = oatt.full_attention(f64(q), f64(k), f64(v), True)
    assert max_err(out, ro) <= TOL_BF16_OUT and max_err(lse, rl) <= TOL_BF16_LSE
    o, l = _device_call(ra, q, k, v, kw)
    assert torch.equal(out, o) and torch.equal(lse, l)


def test_host_path_grouped_32k_bitwise_and_sampled(ra):
    """The 32k GQA zigzag workload, split into KV-head groups whose copies overlap the
    attention: bitwise equal to one device-buffer launch, and sampled rows vs the oracle."""
    from online_softmax_attention_zigzag_gb300.configs import CAUSAL_GQA_S32K as w
    from online_softmax_attention_zigzag_gb300.inputs import make_qkv, sample_rows
    q, k, v = make_qkv(w)
    kw = dict(c=w.c, causal=w.causal, layout=w.layout, kv_block=w.kv_block)
    out, lse = _host_call(ra, q, k, v, kw)
    o, l = _device_call(ra, q, k, v, kw)
    assert torch.equal(out, o) and torch.equal(lse, l)
    hs, ps = sample_rows(w.bhq, w.seq, 512)
    ro, rl = oatt.full_attention_rows(q, k, v, hs.numpy(), ps.numpy(), True)
    assert max_err(out[hs, ps], ro) <= TOL_BF16_OUT and max_err(lse[hs, ps], rl) <= TOL_BF16_LSE


def test_host_path_two_calls_share_workspace(ra):
    """Two calls on one stream reuse one workspace; the second sees none of the first."""
    Hq, Hkv, S, d = 4, 4, 1024, 64
    kw = dict(c=2, causal=1, layout=0, kv_block=512)
    ws = torch.empty(ra.host_workspace_bytes(S, Hq, Hkv, d), dtype=torch.uint8, device=dev())
    res = []
    for seed in (61, 71):
        q, k, v = (_randn((h, S, d), seed + i).pin_memory() for i, h in enumerate((Hq, Hkv, Hkv)))
        out = torch.empty((Hq, S, d), dtype=torch.float32, pin_memory=True)
        lse = torch.empty((Hq, S), dtype=torch.float32, pin_memory=True)
        ra.fwd_host(q, k, v, out, lse, ws, **kw)
        res.append((q, k, v, out, lse))
    assert ra.sync_status() == ra.RA_OK
    for q, k, v, out, lse in res:
        ro, rl = oatt.full_attention(f64(q), f64(k), f64(v), True)
        assert max_err(out, ro) <= TOL_BF16_OUT and max_err(lse, rl) <= TOL_BF16_LSE
