"""The online-softmax correction under stress, through the C ABI against the float64 oracle.

"Ring Attention and Ulysses shard a sequence two different ways..." (section "Ring
Attention: point-to-point rotation...") makes the correction the whole mechanism: when a
block's scores exceed everything seen so far, the running sum and output are rescaled by
e^(old max - new max).  The fused kernel applies that rescale lazily: it keeps a stale
reference max until a row's true max exceeds it by more than 2^8 in log2 units (then P
stays below 2^8 and O needs no rescale otherwise).  Random inputs seldom reach either side
of that threshold, so the inputs here are built to:

* ``rising``: key feature 0 grows by 6 per 128-key tile along every chunk (q feature 0 is
  1), so within each ring block the row max rises by 6 * log2(e) = 8.66 > 8 log2 units at
  every tile and the rescale branch runs on every tile of the block;
* ``held``: key feature 0 is 0 on the first tile of every chunk and 5.46875 elsewhere
  (7.89 log2 units, just under the threshold), so after a rank's first tile the reference
  max is never moved and every later P is about 2^7.89 = 237, the largest the kernel
  allows, summed over thousands of keys.

A small random part on the other features keeps the rows distinct; V is N(0, 1).
"""
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


def _inputs(kind, Hq, Hkv, S, d, n_chunks, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((Hq, S, d), generator=g) * 0.05
    # small enough in "held" that no row's max crosses the threshold: |q.k| off feature 0
    # has a standard deviation of about 0.011 at d = 128
    k = torch.randn((Hkv, S, d), generator=g) * (0.05 if kind == "rising" else 0.02)
    v = torch.randn((Hkv, S, d), generator=g)
    q[..., 0] = 1.0
    m = S // n_chunks
    tile_in_chunk = (torch.arange(S) % m) // 128
    if kind == "rising":
        k[..., 0] = 6.0 * tile_in_chunk.to(torch.float32)
    else:
        k[..., 0] = torch.where(tile_in_chunk == 0, 0.0, 5.46875)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


CASES = [
    # kind, Hq, Hkv, S, d, c, layout, causal
    ("rising", 2, 1, 2048, 128, 4, 0, 0),    # head pairs, 4 tiles per chunk, non-causal
    ("rising", 2, 1, 4096, 128, 4, 1, 1),    # zigzag, causal
    ("rising", 2, 2, 2048, 64, 2, 0, 1),     # position pairs, 8 tiles per chunk
    ("held", 2, 1, 4096, 128, 4, 1, 0),      # zigzag, non-causal: ~4000 keys at P ~ 237
    ("held", 2, 1, 4096, 128, 2, 0, 1),      # contiguous, causal
    ("held", 3, 3, 2048, 64, 4, 1, 1),       # MHA, zigzag, causal
]


@pytest.mark.parametrize("case", CASES)
def test_lazy_rescale_against_oracle(ra, case):
    kind, Hq, Hkv, S, d, c, layout, causal = case
    n_chunks = c * (2 if layout else 1)
    q, k, v = _inputs(kind, Hq, Hkv, S, d, n_chunks, 400 + S + d)
    out, lse = ra.attention(q.to(dev()), k.to(dev()), v.to(dev()), c=c, causal=causal, layout=layout,
                            kv_block=S // n_chunks)
    torch.cuda.synchronize()
    assert ra.sync_status() == ra.RA_OK
    ro, rl = oatt.full_attention(f64(q), f64(k), f64(v), bool(causal))
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    assert max_err(out.cpu(), ro) <= TOL_BF16_OUT, max_err(out.cpu(), ro)
    assert max_err(lse.cpu(), rl) <= TOL_BF16_LSE, max_err(lse.cpu(), rl)


@pytest.mark.parametrize("kind", ["rising", "held"])
def test_lazy_rescale_per_hop_path(ra, kind):
    """The same inputs through one partial per ring message and the merge kernel: each
    message's kernel launch starts its own reference max, and the merge rescales."""
    Hq, Hkv, S, d, c, layout, causal = 2, 1, 2048, 128, 2, 1, 1
    q, k, v = _inputs(kind, Hq, Hkv, S, d, 2 * c, 431)
    kvb = 256
    qr, kr, vr = (torch.empty(x.shape, dtype=x.dtype, device=dev()) for x in (q, k, v))
    for src, dst in ((q, qr), (k, kr), (v, vr)):
        ra.permute(src.to(dev()), dst, c=c, layout=layout, inverse=0)
    o_run = torch.zeros((Hq, S, d), dtype=torch.float32, device=dev())
    l_run = torch.full((Hq, S), -float("inf"), dtype=torch.float32, device=dev())
    op, lp = torch.empty_like(o_run), torch.empty_like(l_run)
    for hop in range(c):
        for sub in range((S // c) // kvb):
            ra.fwd_hop(qr, kr, vr, op, lp, c=c, causal=causal, layout=layout, kv_block=kvb, hop=hop, sub=sub)
            ra.merge(o_run, l_run, op, lp)
    out, lse = torch.empty_like(o_run), torch.empty_like(l_run)
    ra.permute(o_run, out, c=c, layout=layout, inverse=1)
    ra.permute(l_run, lse, c=c, layout=layout, inverse=1)
    torch.cuda.synchronize()
    assert ra.sync_status() == ra.RA_OK
    ro, rl = oatt.full_attention(f64(q), f64(k), f64(v), True)
    assert max_err(out.cpu(), ro) <= TOL_BF16_OUT
    assert max_err(lse.cpu(), rl) <= TOL_BF16_LSE
