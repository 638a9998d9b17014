"""Ulysses on one GPU (ringattn_relayout, ringattn_ulysses_fwd) against the oracle
("Ring Attention and Ulysses shard a sequence two different ways...", section "Ulysses:
an all-to-all relayout instead of a rotation").  Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import layout as olay
from oracle import ulysses as oul
from tests.gpu_util import TOL_BF16_LSE, TOL_BF16_OUT, dev, f64, max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    from online_softmax_attention_zigzag_gb300 import ringattn
    ringattn.lib()
    torch.cuda.set_device(0)
    return ringattn


def _randn(shape, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(dtype)


def _seq(x, S, c, layout):
    """[H, S, ...] natural -> sequence-sharded [S, H, ...] (rank-major tokens), by indexing."""
    order = torch.from_numpy(olay.rank_major_order(S, c, layout))
    return x[:, order].transpose(0, 1).contiguous()


def _bits(t):
    """Raw bit pattern as int64 numpy (exact for every dtype used here)."""
    view = {2: torch.int16, 4: torch.int32}[t.element_size()]
    return t.contiguous().view(view).to(torch.int64).numpy()


@pytest.mark.parametrize("S,H,row_shape,dtype,c,layout", [
    (4096, 8, (128,), torch.bfloat16, 4, 1),     # q/k/v rows, 16-byte vectors
    (2304, 6, (128,), torch.float32, 3, 1),      # out rows
    (1536, 4, (64,), torch.bfloat16, 3, 0),      # d = 64, contiguous
    (2048, 16, (), torch.float32, 8, 1),         # lse: 4-byte rows
    (96, 3, (3,), torch.float32, 3, 1),          # 12-byte rows: 4-byte vectors, tiny chunks
    (40, 2, (8,), torch.bfloat16, 5, 0),         # 16-byte rows, chunk of 8 tokens
])
def test_relayout_bit_exact_both_directions(ra, S, H, row_shape, dtype, c, layout):
    x_seq = _randn((S, H) + row_shape, 91 + S + H, dtype)
    heads = torch.empty((H, S) + row_shape, dtype=dtype, device=dev())
    ra.relayout(x_seq.to(dev()), heads, c=c, layout=layout, to_heads=1)
    back = torch.empty((S, H) + row_shape, dtype=dtype, device=dev())
    ra.relayout(heads, back, c=c, layout=layout, to_heads=0)
    assert ra.sync_status() == ra.RA_OK
    # the oracle's message-by-message all-to-all, one rank per head group when H % c == 0,
    # else every head on one receiver (the placement does not depend on the split)
    bits = _bits(x_seq).reshape(S, H, -1)
    split = H % c == 0
    heads_of = (lambda r: np.arange(r * (H // c), (r + 1) * (H // c))) if split else \
        (lambda r: np.arange(H) if r == 0 else np.arange(0))
    parts = oul.seq_to_heads(oul.split_shards(bits, c), heads_of, S, c, layout)
    want = np.concatenate([p for p in parts if p.shape[0]]).astype(np.int64)
    assert np.array_equal(_bits(heads.cpu()).reshape(H, S, -1), want)
    assert torch.equal(back.cpu(), x_seq)


def _ulysses(ra, q, k, v, c, layout, causal):
    Hq, S, d = q.shape
    Hkv = k.shape[0]
    qs, ks, vs = (_seq(x, S, c, layout).to(dev()) for x in (q, k, v))
    out = torch.full((S, Hq, d), float("nan"), dtype=torch.float32, device=dev())
    lse = torch.full((S, Hq), float("nan"), dtype=torch.float32, device=dev())
    ws = torch.empty(ra.host_workspace_bytes(S, Hq, Hkv, d), dtype=torch.uint8, device=dev())
    ra.ulysses_fwd(qs, ks, vs, out, lse, ws, c=c, causal=causal, layout=layout)
    assert ra.sync_status() == ra.RA_OK
    return qs.cpu(), ks.cpu(), vs.cpu(), out.cpu(), lse.cpu()


@pytest.mark.parametrize("Hq,Hkv,S,d,c,layout,causal", [
    (8, 2, 2048, 128, 4, 1, 1),     # GQA, zigzag, causal
    (8, 2, 2048, 128, 8, 1, 1),     # more ranks than KV heads: a KV head serves 4 ranks
    (4, 4, 1024, 64, 2, 0, 1),      # MHA d = 64, contiguous
    (6, 3, 768, 128, 3, 1, 0),      # non-causal, g = 2, c = 3
])
def test_ulysses_vs_oracle(ra, Hq, Hkv, S, d, c, layout, causal):
    q, k, v = _randn((Hq, S, d), 101), _randn((Hkv, S, d), 102), _randn((Hkv, S, d), 103)
    qs, ks, vs, out, lse = _ulysses(ra, q, k, v, c, layout, causal)
    ro, rl = oul.ulysses_attention(f64(qs), f64(ks), f64(vs), c, layout, bool(causal))
    assert max_err(out, ro) <= TOL_BF16_OUT, max_err(out, ro)
    assert max_err(lse, rl) <= TOL_BF16_LSE, max_err(lse, rl)


def test_ulysses_32k_sampled_and_equal_to_ring(ra):
    """The 32k GQA zigzag workload: sampled rows against the oracle, every row against
    the ring (rounding only: the two visit keys in different orders)."""
    from online_softmax_attention_zigzag_gb300.configs import CAUSAL_GQA_S32K as w
    from online_softmax_attention_zigzag_gb300.inputs import make_qkv, sample_rows
    q, k, v = make_qkv(w)
    S = w.seq
    _, _, _, out, lse = _ulysses(ra, q, k, v, w.c, w.layout, w.causal)
    order = olay.rank_major_order(S, w.c, w.layout)
    hs, ps = sample_rows(w.bhq, S, 1024)
    tok = torch.from_numpy(np.argsort(order)[ps.numpy()])  # rank-major token of each sampled position
    ro, rl = oatt.full_attention_rows(q, k, v, hs.numpy(), ps.numpy(), True)
    assert max_err(out[tok, hs], ro) <= TOL_BF16_OUT
    assert max_err(lse[tok, hs], rl) <= TOL_BF16_LSE
    on = torch.empty((w.bhq, S, w.d), dtype=torch.float32, device=dev())
    ln = torch.empty((w.bhq, S), dtype=torch.float32, device=dev())
    ra.fwd_natural(q.to(dev()), k.to(dev()), v.to(dev()), on, ln, c=w.c, causal=1, layout=w.layout,
                   kv_block=w.kv_block)
    assert ra.sync_status() == ra.RA_OK
    ring_seq_o = on.cpu()[:, order].transpose(0, 1)
    ring_seq_l = ln.cpu()[:, order].transpose(0, 1)
    assert max_err(out, ring_seq_o) <= TOL_BF16_OUT and max_err(lse, ring_seq_l) <= TOL_BF16_LSE
