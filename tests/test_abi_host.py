"""The C ABI on the host (no GPU needed): exports, argument validation, host-only work counts."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import work as oracle_work

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ra():
    from online_softmax_attention_zigzag_gb300 import ringattn
    if not os.path.exists(ringattn.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return ringattn


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*(?:int|const char\*)\s+(ringattn_\w+)\s*\(", src, re.M))
    return names


def test_library_exports_every_declared_symbol(ra):
    declared = _declared()
    assert len(declared) >= 10
    L = ra.lib()
    for name in declared:
        assert hasattr(L, name), name
    assert set(ra.EXPORTS) == declared


def test_check_build_exports_the_same_symbols(ra):
    """libringattn_check.so (compiled with -DRA_CHECK) is the same ABI."""
    path = os.path.join(os.path.dirname(ra.LIB_PATH), "libringattn_check.so")
    assert os.path.exists(path), "build() makes the check build too"
    L = ctypes.CDLL(path)
    for name in _declared():
        assert hasattr(L, name), name
    L.ringattn_strerror.restype = ctypes.c_char_p
    assert b"index check" in L.ringattn_strerror(-6)


def test_strerror(ra):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert ra.strerror(code) not in ("", "unknown status")
    assert ra.strerror(12345) == "unknown status"


# Fake, 16-byte aligned, never-dereferenced device addresses: every call below must be
# rejected by host validation before any device is touched.
P = ctypes.c_void_p(0x10000)
P2 = ctypes.c_void_p(0x20000)
NUL = ctypes.c_void_p(0)
S0 = ctypes.c_void_p(0)


def _fwd(ra, *args, fn="ringattn_fwd"):
    return getattr(ra.lib(), fn)(*args)


@pytest.mark.parametrize("case,expect", [
    (dict(S=4096, Hq=8, Hkv=3, d=64, c=4, causal=1, layout=1, kvb=512), -1),   # Hq % Hkv
    (dict(S=4004, Hq=8, Hkv=8, d=64, c=4, causal=1, layout=1, kvb=500), -1),   # S % 2c
    (dict(S=4096, Hq=8, Hkv=8, d=64, c=4, causal=2, layout=1, kvb=512), -1),   # causal flag
    (dict(S=4096, Hq=8, Hkv=8, d=64, c=4, causal=1, layout=3, kvb=512), -1),   # layout flag
    (dict(S=4096, Hq=8, Hkv=8, d=64, c=0, causal=1, layout=1, kvb=512), -1),   # c
    (dict(S=4096, Hq=8, Hkv=8, d=64, c=4, causal=1, layout=1, kvb=384), -1),   # kv_block divides chunk
    (dict(S=4096, Hq=8, Hkv=8, d=96, c=4, causal=1, layout=1, kvb=512), -2),   # d on the bf16 path
    (dict(S=4096 + 64 * 8, Hq=8, Hkv=8, d=64, c=4, causal=1, layout=1, kvb=64), -2),  # chunk % 128
    (dict(S=0, Hq=8, Hkv=8, d=64, c=4, causal=1, layout=1, kvb=512), -1),
])
def test_fwd_rejects_bad_arguments(ra, case, expect):
    c = case
    assert _fwd(ra, P, P, P, P2, P2, c["S"], c["Hq"], c["Hkv"], c["d"], c["c"], c["causal"], c["layout"],
                c["kvb"], S0) == expect


def test_fwd_rejects_null_and_misaligned(ra):
    args = [4096, 8, 8, 64, 4, 1, 1, 512, S0]
    assert _fwd(ra, NUL, P, P, P2, P2, *args) == -1
    assert _fwd(ra, P, P, P, P2, NUL, *args) == -1
    assert _fwd(ra, ctypes.c_void_p(0x10008), P, P, P2, P2, *args) == -1


def test_hop_rejects_bad_hop_and_sub(ra):
    L = ra.lib()
    base = [P, P, P, P2, P2, 4096, 8, 8, 64, 4, 1, 1, 512]
    assert L.ringattn_fwd_hop(*base, 4, 0, S0) == -1       # hop >= c
    assert L.ringattn_fwd_hop(*base, -1, 0, S0) == -1
    assert L.ringattn_fwd_hop(*base, 0, 2, S0) == -1       # (S/c)/kv_block = 2 messages
    assert L.ringattn_fwd_hop_f32(*base, 0, -1, S0) == -1


def test_rank_rejects_bad_rank(ra):
    L = ra.lib()
    base = [P, P, P, P2, P2, 4096, 8, 8, 64, 4, 1, 1, 512]
    assert L.ringattn_fwd_rank(*base, 4, S0) == -1          # rank >= c
    assert L.ringattn_fwd_rank(*base, -1, S0) == -1
    assert L.ringattn_fwd_rank(P, P, P, P2, P2, 4096, 8, 3, 64, 4, 1, 1, 512, 0, S0) == -1  # geometry too


def test_docmask_rejects(ra):
    L = ra.lib()
    D1, D2 = ctypes.c_void_p(0x30000), ctypes.c_void_p(0x40000)
    geo = [4096, 8, 2, 128, 4, 1]
    assert L.ringattn_fwd_docmask(P, P, P, P2, P2, NUL, D2, *geo, S0) == -1          # null ids
    assert L.ringattn_fwd_docmask(P, P, P, P2, P2, D1, D1, *geo, S0) == -1           # scratch aliases ids
    assert L.ringattn_fwd_docmask(P, P, P, P2, P2, ctypes.c_void_p(0x30002), D2, *geo, S0) == -1  # alignment
    assert L.ringattn_fwd_docmask(P, P, P, P2, P2, D1, D2, 4100, 8, 2, 128, 4, 1, S0) == -1       # S % 2c
    assert L.ringattn_fwd_docmask(P, P, P, P2, P2, D1, D2, 4096, 8, 3, 128, 4, 1, S0) == -1       # Hq % Hkv
    assert L.ringattn_fwd_docmask(P, P, P, P2, P2, D1, D2, 4096, 8, 2, 96, 4, 1, S0) == -2        # d
    assert L.ringattn_fwd_docmask(P, P, P, P2, P2, D1, D2, 4096, 8, 2, 128, 4, 2, S0) == -1       # layout


def test_docmask_noalloc_rejects(ra):
    L = ra.lib()
    D1 = ctypes.c_void_p(0x30000)
    hdr = open(os.path.join(ROOT, "include", "ringattn.h")).read()
    assert int(re.search(r"#define RINGATTN_DOCMASK_NOALLOC_MAX_S (\d+)", hdr).group(1)) == ra.DOCMASK_NOALLOC_MAX_S
    big = ra.DOCMASK_NOALLOC_MAX_S + 256
    assert L.ringattn_fwd_docmask_noalloc(P, P, P, P2, P2, NUL, 4096, 8, 2, 128, 4, 1, S0) == -1  # null ids
    assert L.ringattn_fwd_docmask_noalloc(P, P, P, P2, P2, ctypes.c_void_p(0x30002), 4096, 8, 2, 128, 4, 1,
                                          S0) == -1                                                # alignment
    assert L.ringattn_fwd_docmask_noalloc(P, P, P, P2, P2, D1, big, 8, 2, 128, 4, 1, S0) == -2     # beyond scratch
    assert L.ringattn_fwd_docmask_noalloc(P, P, P, P2, P2, D1, 4100, 8, 2, 128, 4, 1, S0) == -1    # S % 2c
    assert L.ringattn_fwd_docmask_noalloc(P, P, P, P2, P2, D1, 4096, 8, 2, 128, 4, 2, S0) == -1    # layout


def test_host_path_workspace_and_rejects(ra):
    L = ra.lib()
    n = ctypes.c_longlong(0)
    assert L.ringattn_host_workspace_bytes(1000, 3, 1, 64, ctypes.byref(n)) == 0
    # q, k, v bf16 and out, lse fp32, each rounded up to 256 bytes
    sizes = [2 * 3 * 1000 * 64, 2 * 1000 * 64, 2 * 1000 * 64, 4 * 3 * 1000 * 64, 4 * 3 * 1000]
    assert n.value == sum((x + 255) // 256 * 256 for x in sizes)
    assert L.ringattn_host_workspace_bytes(0, 3, 1, 64, ctypes.byref(n)) == -1
    assert L.ringattn_host_workspace_bytes(1000, 3, 1, 64, NUL) == -1
    need = ra.host_workspace_bytes(4096, 8, 2, 128)
    W = ctypes.c_void_p(0x100000)
    geo = [4096, 8, 2, 128, 4, 1, 1, 512]
    assert L.ringattn_fwd_host(NUL, P, P, P2, P2, *geo, W, need, S0) == -1                   # null input
    assert L.ringattn_fwd_host(P, P, P, P2, P2, *geo, NUL, need, S0) == -1                   # null workspace
    assert L.ringattn_fwd_host(P, P, P, P2, P2, *geo, ctypes.c_void_p(0x100010), need, S0) == -1  # alignment
    assert L.ringattn_fwd_host(P, P, P, P2, P2, *geo, W, need - 1, S0) == -1                 # too small
    assert L.ringattn_fwd_host(P, P, P, P2, P2, *geo, W, -5, S0) == -1
    assert L.ringattn_fwd_host(P, P, P, P2, P2, 4096, 8, 3, 128, 4, 1, 1, 512, W, need, S0) == -1  # Hq % Hkv
    assert L.ringattn_fwd_host(P, P, P, P2, P2, 4096, 8, 2, 96, 4, 1, 1, 512, W, need, S0) == -2   # d


def test_f32_rejects(ra):
    L = ra.lib()
    assert L.ringattn_fwd_f32(P, P, P, P2, P2, 12, 1, 1, 129, 3, 0, 0, 4, S0) == -2   # d > 128
    assert L.ringattn_fwd_f32(P, P, P, P2, P2, 12, 1, 1, 8, 3, 0, 0, 3, S0) == -1     # kv_block
    assert L.ringattn_fwd_f32(P, P, P, P2, P2, 12, 1, 1, 8, 5, 0, 0, 1, S0) == -1     # S % c


def test_merge_and_permute_reject(ra):
    L = ra.lib()
    assert L.ringattn_merge(P, P, P2, P2, -1, 128, S0) == -1
    assert L.ringattn_merge(P, P, P2, P2, 10, 0, S0) == -1
    assert L.ringattn_merge(NUL, P, P2, P2, 10, 64, S0) == -1
    assert L.ringattn_merge(NUL, NUL, NUL, NUL, 0, 64, S0) == 0     # nothing to do
    assert L.ringattn_permute(P, P, 16, 1, 4, 2, 1, 0, S0) == -1     # in place
    assert L.ringattn_permute(P, ctypes.c_void_p(0x10010), 16, 1, 4, 2, 1, 0, S0) == -1  # overlap
    assert L.ringattn_permute(P, P2, 15, 1, 4, 2, 1, 0, S0) == -1    # S % 2c
    assert L.ringattn_permute(P, P2, 16, 1, 4, 2, 1, 2, S0) == -1    # inverse flag
    assert L.ringattn_selftest_timeout(10, S0) == -1


@pytest.mark.parametrize("S,c,causal,layout,tile", [
    (1024, 8, 1, 0, 128), (1024, 8, 1, 1, 128), (4096, 4, 1, 1, 128), (4096, 4, 1, 0, 128),
    (96, 3, 1, 1, 4), (96, 3, 0, 1, 4), (48, 3, 1, 1, 5), (4096, 4, 0, 0, 128), (32768, 8, 1, 1, 128),
])
def test_rank_work_matches_oracle(ra, S, c, causal, layout, tile):
    u, p, t = ra.rank_work(S, c, causal, layout, tile)
    ou, op, ot = oracle_work.rank_work(S, c, bool(causal), layout, tile)
    assert np.array_equal(u, ou) and np.array_equal(p, op) and np.array_equal(t, ot)


def test_rank_work_zigzag_balanced_contiguous_skewed(ra):
    u, p, t = ra.rank_work(32768, 8, 1, 1, 128)
    assert len(set(u)) == 1 and u[0] == 17 and len(set(p)) == 1 and len(set(t)) == 1
    u, p, t = ra.rank_work(32768, 8, 1, 0, 128)
    assert list(u) == list(range(1, 9))


def test_binding_rejects_a_tensor_on_another_device(ra, monkeypatch):
    """The binding passes raw device pointers to kernels launched on the current device, so a
    tensor on another device is refused before any call (stand-in tensors: no GPU here)."""
    from unittest import mock
    import torch

    def fake(index):
        t = mock.MagicMock(spec=torch.Tensor)
        t.is_cuda = True
        t.device = torch.device("cuda", index)
        t.dtype = torch.float32
        t.is_contiguous.return_value = True
        t.data_ptr.return_value = 4096
        return t

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    assert ra._dev(fake(0), "x", torch.float32).value == 4096
    with pytest.raises(ValueError, match="current device is cuda:0"):
        ra._dev(fake(1), "x", torch.float32)
