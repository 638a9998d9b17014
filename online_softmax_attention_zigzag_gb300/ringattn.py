"""Thin Python binding of libringattn.so (C ABI in include/ringattn.h).

Argument marshalling only: every function checks shapes/dtypes/devices of the
torch tensors it is given, passes their device pointers and sizes to the C
entry point of the same name, and raises :class:`RingAttnError` on a non-zero
status.  PyTorch provides device memory and streams; all computation happens in
the library's CUDA kernels.  There is no fallback: if the library is missing
or the device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# RINGATTN_CHECK=1 loads the check build (index checks in the kernels, RA_ERR_BOUNDS);
# same ABI, same results
LIB_PATH = os.path.join(_PKG, "libringattn_check.so" if os.environ.get("RINGATTN_CHECK") == "1"
                        else "libringattn.so")

RA_OK = 0
RA_ERR_INVALID_ARG = -1
RA_ERR_UNSUPPORTED = -2
RA_ERR_ARCH = -3
RA_ERR_CUDA = -4
RA_ERR_TIMEOUT = -5
RA_ERR_BOUNDS = -6

EXPORTS = (
    "ringattn_fwd", "ringattn_fwd_natural", "ringattn_fwd_f32", "ringattn_fwd_hop",
    "ringattn_fwd_hop_f32", "ringattn_merge", "ringattn_permute", "ringattn_rank_work",
    "ringattn_sync_status", "ringattn_selftest_timeout", "ringattn_strerror", "ringattn_last_timeout",
    "ringattn_fwd_rank", "ringattn_fwd_docmask", "ringattn_fwd_docmask_noalloc",
    "ringattn_fwd_host", "ringattn_host_workspace_bytes", "ringattn_relayout", "ringattn_ulysses_fwd",
    "ringattn_bwd", "ringattn_bwd_natural",
)

# Longest sequence ringattn_fwd_docmask_noalloc takes (its static scratch, int32 [S]).
DOCMASK_NOALLOC_MAX_S = 262144


class RingAttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {code} ({strerror(code)})")


_lib = None

_P, _I, _LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
_ATTN = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I]


def lib() -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                "or python -m online_softmax_attention_zigzag_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "ringattn_fwd": _ATTN + [_P],
            "ringattn_fwd_natural": _ATTN + [_P],
            "ringattn_fwd_rank": _ATTN + [_I, _P],
            "ringattn_fwd_docmask": [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P],
            "ringattn_fwd_docmask_noalloc": [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P],
            "ringattn_fwd_host": _ATTN + [_P, _LL, _P],
            "ringattn_host_workspace_bytes": [_I, _I, _I, _I, _P],
            "ringattn_relayout": [_P, _P, _I, _I, _I, _I, _I, _I, _P],
            "ringattn_bwd": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P],
            "ringattn_bwd_natural": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P],
            "ringattn_ulysses_fwd": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _LL, _P],
            "ringattn_fwd_f32": _ATTN + [_P],
            "ringattn_fwd_hop": _ATTN + [_I, _I, _P],
            "ringattn_fwd_hop_f32": _ATTN + [_I, _I, _P],
            "ringattn_merge": [_P, _P, _P, _P, _LL, _I, _P],
            "ringattn_permute": [_P, _P, _I, _I, _I, _I, _I, _I, _P],
            "ringattn_rank_work": [_I, _I, _I, _I, _I, _P, _P, _P],
            "ringattn_sync_status": [_P],
            "ringattn_selftest_timeout": [_LL, _P],
            "ringattn_last_timeout": [_P],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = _I
        L.ringattn_strerror.argtypes = [_I]
        L.ringattn_strerror.restype = ctypes.c_char_p
        _lib = L
    return _lib


def strerror(code: int) -> str:
    try:
        return lib().ringattn_strerror(int(code)).decode()
    except Exception:  # the library itself may be missing
        return "unknown"


def _check(fn: str, code: int) -> None:
    if code != RA_OK:
        raise RingAttnError(fn, code)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        # the library launches on the current device; another device's pointer would reach
        # its kernels as a foreign address
        raise ValueError(f"{name} is on {t.device}, but the current device is "
                         f"cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _attn_args(q, k, v, out, lse, in_dtype):
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be [H, S, d]")
    Hq, S, d = q.shape
    Hkv = k.shape[0]
    if tuple(k.shape) != (Hkv, S, d) or tuple(v.shape) != (Hkv, S, d):
        raise ValueError("k and v must be [Hkv, S, d] with q's S and d")
    if tuple(out.shape) != (Hq, S, d) or tuple(lse.shape) != (Hq, S):
        raise ValueError("out must be [Hq, S, d] and lse [Hq, S]")
    ptrs = [_dev(q, "q", in_dtype), _dev(k, "k", in_dtype), _dev(v, "v", in_dtype),
            _dev(out, "out", torch.float32), _dev(lse, "lse", torch.float32)]
    return ptrs, S, Hq, Hkv, d


def fwd(q, k, v, out, lse, *, c, causal, layout, kv_block, stream=None) -> None:
    """ringattn_fwd: bf16 rank-major q [Hq,S,d], k/v [Hkv,S,d] -> fp32 out, lse."""
    ptrs, S, Hq, Hkv, d = _attn_args(q, k, v, out, lse, torch.bfloat16)
    _check("ringattn_fwd", lib().ringattn_fwd(*ptrs, S, Hq, Hkv, d, c, int(causal), layout, kv_block,
                                              ctypes.c_void_p(_stream(stream))))


def fwd_rank(q, k, v, out, lse, *, c, causal, layout, kv_block, rank, stream=None) -> None:
    """ringattn_fwd_rank: as :func:`fwd`, writing only the rows virtual rank ``rank`` holds."""
    ptrs, S, Hq, Hkv, d = _attn_args(q, k, v, out, lse, torch.bfloat16)
    _check("ringattn_fwd_rank", lib().ringattn_fwd_rank(*ptrs, S, Hq, Hkv, d, c, int(causal), layout, kv_block,
                                                        int(rank), _stream(stream)))


def fwd_docmask(q, k, v, out, lse, doc_id, doc_start, *, c, layout, stream=None) -> None:
    """ringattn_fwd_docmask: all-gathered K/V, causal inside each document of ``doc_id``
    (int32 [S], natural order, non-decreasing); ``doc_start`` is int32 [S] scratch."""
    ptrs, S, Hq, Hkv, d = _attn_args(q, k, v, out, lse, torch.bfloat16)
    for t, name in ((doc_id, "doc_id"), (doc_start, "doc_start")):
        if tuple(t.shape) != (S,):
            raise ValueError(f"{name} must be [S]")
    ptrs += [_dev(doc_id, "doc_id", torch.int32), _dev(doc_start, "doc_start", torch.int32)]
    _check("ringattn_fwd_docmask", lib().ringattn_fwd_docmask(*ptrs, S, Hq, Hkv, d, c, layout, _stream(stream)))


def fwd_docmask_noalloc(q, k, v, out, lse, doc_id, *, c, layout, stream=None) -> None:
    """ringattn_fwd_docmask_noalloc: :func:`fwd_docmask` without the scratch argument, for
    callers that cannot allocate device memory; the document starts live in the library's
    static device array, shared by every call (order overlapping calls on one stream)."""
    ptrs, S, Hq, Hkv, d = _attn_args(q, k, v, out, lse, torch.bfloat16)
    if tuple(doc_id.shape) != (S,):
        raise ValueError("doc_id must be [S]")
    if S > DOCMASK_NOALLOC_MAX_S:
        raise ValueError(f"S = {S} exceeds the static scratch of ringattn_fwd_docmask_noalloc "
                         f"({DOCMASK_NOALLOC_MAX_S} positions); use fwd_docmask with caller-owned scratch")
    ptrs.append(_dev(doc_id, "doc_id", torch.int32))
    _check("ringattn_fwd_docmask_noalloc",
           lib().ringattn_fwd_docmask_noalloc(*ptrs, S, Hq, Hkv, d, c, layout, _stream(stream)))


def host_workspace_bytes(S: int, Hq: int, Hkv: int, d: int) -> int:
    """ringattn_host_workspace_bytes (host only)."""
    n = ctypes.c_longlong(0)
    _check("ringattn_host_workspace_bytes", lib().ringattn_host_workspace_bytes(S, Hq, Hkv, d, ctypes.byref(n)))
    return n.value


def _host(t: torch.Tensor, name: str, dtype):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def fwd_host(q_h, k_h, v_h, out_h, lse_h, workspace, *, c, causal, layout, kv_block, stream=None) -> None:
    """ringattn_fwd_host: natural-order HOST tensors (pin them for overlap) in, HOST out and
    lse out; ``workspace`` is a CUDA uint8 tensor of at least :func:`host_workspace_bytes`.
    Asynchronous on ``stream``: synchronise it before reading out_h / lse_h."""
    if q_h.dim() != 3 or k_h.dim() != 3 or v_h.dim() != 3:
        raise ValueError("q, k, v must be [H, S, d]")
    Hq, S, d = q_h.shape
    Hkv = k_h.shape[0]
    if tuple(k_h.shape) != (Hkv, S, d) or tuple(v_h.shape) != (Hkv, S, d):
        raise ValueError("k and v must be [Hkv, S, d] with q's S and d")
    if tuple(out_h.shape) != (Hq, S, d) or tuple(lse_h.shape) != (Hq, S):
        raise ValueError("out must be [Hq, S, d] and lse [Hq, S]")
    ptrs = [_host(q_h, "q", torch.bfloat16), _host(k_h, "k", torch.bfloat16), _host(v_h, "v", torch.bfloat16),
            _host(out_h, "out", torch.float32), _host(lse_h, "lse", torch.float32)]
    ws = _dev(workspace, "workspace")
    _check("ringattn_fwd_host", lib().ringattn_fwd_host(
        *ptrs, S, Hq, Hkv, d, c, causal, layout, kv_block, ws, workspace.numel() * workspace.element_size(),
        _stream(stream)))


def relayout(src, dst, *, c, layout, to_heads, stream=None) -> None:
    """ringattn_relayout: to_heads=1 moves sequence-sharded [S, H, ...] (rank-major tokens)
    to head-sharded [H, S, ...] (natural tokens); to_heads=0 the reverse."""
    if src.dtype != dst.dtype or src.numel() != dst.numel():
        raise ValueError("src and dst must have the same dtype and size")
    if src.dim() < 2 or dst.dim() < 2:
        raise ValueError("src and dst must be at least [S, H] / [H, S]")
    S, H = (src.shape[0], src.shape[1]) if to_heads else (src.shape[1], src.shape[0])
    if (tuple(dst.shape[:2]) != ((H, S) if to_heads else (S, H))) or dst.shape[2:] != src.shape[2:]:
        raise ValueError("dst must be src with its first two axes swapped")
    row_bytes = src.element_size() * (src.numel() // max(1, H * S))
    _check("ringattn_relayout", lib().ringattn_relayout(
        _dev(src, "src"), _dev(dst, "dst"), S, H, row_bytes, c, layout, int(to_heads), _stream(stream)))


def ulysses_fwd(q_seq, k_seq, v_seq, out_seq, lse_seq, workspace, *, c, causal, layout, stream=None) -> None:
    """ringattn_ulysses_fwd: sequence-sharded q [S, Hq, d], k, v [S, Hkv, d] bf16 in;
    out [S, Hq, d], lse [S, Hq] fp32 out; workspace a CUDA uint8 tensor of at least
    :func:`host_workspace_bytes` (S, Hq, Hkv, d)."""
    if q_seq.dim() != 3 or k_seq.dim() != 3 or v_seq.dim() != 3:
        raise ValueError("q, k, v must be [S, H, d]")
    S, Hq, d = q_seq.shape
    Hkv = k_seq.shape[1]
    if tuple(k_seq.shape) != (S, Hkv, d) or tuple(v_seq.shape) != (S, Hkv, d):
        raise ValueError("k and v must be [S, Hkv, d] with q's S and d")
    if tuple(out_seq.shape) != (S, Hq, d) or tuple(lse_seq.shape) != (S, Hq):
        raise ValueError("out must be [S, Hq, d] and lse [S, Hq]")
    ptrs = [_dev(q_seq, "q", torch.bfloat16), _dev(k_seq, "k", torch.bfloat16), _dev(v_seq, "v", torch.bfloat16),
            _dev(out_seq, "out", torch.float32), _dev(lse_seq, "lse", torch.float32)]
    _check("ringattn_ulysses_fwd", lib().ringattn_ulysses_fwd(
        *ptrs, S, Hq, Hkv, d, c, causal, layout, _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def bwd(q, k, v, out, lse, dout, dq, dk, dv, delta, *, c, causal, layout, kv_block, stream=None,
        natural=False) -> None:
    """ringattn_bwd (rank-major tensors) or, with natural=True, ringattn_bwd_natural
    (natural order): gradients of the forward.  q, dout [Hq, S, d] and k, v [Hkv, S, d] bf16;
    out [Hq, S, d], lse [Hq, S] fp32 from the forward; dq, dk, dv fp32 like q, k, v; delta
    [Hq, S] fp32 scratch."""
    ptrs, S, Hq, Hkv, d = _attn_args(q, k, v, out, lse, torch.bfloat16)
    if tuple(dout.shape) != (Hq, S, d) or tuple(dq.shape) != (Hq, S, d):
        raise ValueError("dout and dq must be [Hq, S, d]")
    if tuple(dk.shape) != (Hkv, S, d) or tuple(dv.shape) != (Hkv, S, d) or tuple(delta.shape) != (Hq, S):
        raise ValueError("dk, dv must be [Hkv, S, d] and delta [Hq, S]")
    ptrs += [_dev(dout, "dout", torch.bfloat16), _dev(dq, "dq", torch.float32), _dev(dk, "dk", torch.float32),
             _dev(dv, "dv", torch.float32), _dev(delta, "delta", torch.float32)]
    name = "ringattn_bwd_natural" if natural else "ringattn_bwd"
    _check(name, getattr(lib(), name)(*ptrs, S, Hq, Hkv, d, c, causal, layout, kv_block, _stream(stream)))


def fwd_natural(q, k, v, out, lse, *, c, causal, layout, kv_block, stream=None) -> None:
    """ringattn_fwd_natural: as :func:`fwd` with every tensor in natural order."""
    ptrs, S, Hq, Hkv, d = _attn_args(q, k, v, out, lse, torch.bfloat16)
    _check("ringattn_fwd_natural", lib().ringattn_fwd_natural(
        *ptrs, S, Hq, Hkv, d, c, int(causal), layout, kv_block, ctypes.c_void_p(_stream(stream))))


def fwd_f32(q, k, v, out, lse, *, c, causal, layout, kv_block, stream=None) -> None:
    """ringattn_fwd_f32: fp32 rank-major inputs."""
    ptrs, S, Hq, Hkv, d = _attn_args(q, k, v, out, lse, torch.float32)
    _check("ringattn_fwd_f32", lib().ringattn_fwd_f32(*ptrs, S, Hq, Hkv, d, c, int(causal), layout,
                                                      kv_block, ctypes.c_void_p(_stream(stream))))


def fwd_hop(q, k, v, o_part, lse_part, *, c, causal, layout, kv_block, hop, sub, stream=None) -> None:
    """ringattn_fwd_hop: the partial of one ring message (bf16 inputs)."""
    ptrs, S, Hq, Hkv, d = _attn_args(q, k, v, o_part, lse_part, torch.bfloat16)
    _check("ringattn_fwd_hop", lib().ringattn_fwd_hop(*ptrs, S, Hq, Hkv, d, c, int(causal), layout,
                                                      kv_block, hop, sub, ctypes.c_void_p(_stream(stream))))


def fwd_hop_f32(q, k, v, o_part, lse_part, *, c, causal, layout, kv_block, hop, sub, stream=None) -> None:
    """ringattn_fwd_hop_f32: the partial of one ring message (fp32 inputs)."""
    ptrs, S, Hq, Hkv, d = _attn_args(q, k, v, o_part, lse_part, torch.float32)
    _check("ringattn_fwd_hop_f32", lib().ringattn_fwd_hop_f32(
        *ptrs, S, Hq, Hkv, d, c, int(causal), layout, kv_block, hop, sub, ctypes.c_void_p(_stream(stream))))


def merge(o_run, lse_run, o_part, lse_part, stream=None) -> None:
    """ringattn_merge: fold (o_part, lse_part) into (o_run, lse_run) in place."""
    d = o_run.shape[-1]
    rows = lse_run.numel()
    if o_run.numel() != rows * d or o_part.shape != o_run.shape or lse_part.shape != lse_run.shape:
        raise ValueError("o_* must be [..., d] with one lse per row")
    _check("ringattn_merge", lib().ringattn_merge(
        _dev(o_run, "o_run", torch.float32), _dev(lse_run, "lse_run", torch.float32),
        _dev(o_part, "o_part", torch.float32), _dev(lse_part, "lse_part", torch.float32),
        rows, d, ctypes.c_void_p(_stream(stream))))


def permute(src, dst, *, c, layout, inverse, stream=None) -> None:
    """ringattn_permute: src/dst [H, S, ...] contiguous, same shape and dtype."""
    if src.shape != dst.shape or src.dtype != dst.dtype:
        raise ValueError("src and dst must have the same shape and dtype")
    H, S = src.shape[0], src.shape[1]
    row_bytes = src.element_size() * (src.numel() // max(1, H * S))
    _check("ringattn_permute", lib().ringattn_permute(
        _dev(src, "src"), _dev(dst, "dst"), S, H, row_bytes, c, layout, int(inverse),
        ctypes.c_void_p(_stream(stream))))


def rank_work(S: int, c: int, causal: int, layout: int, tile: int = 128):
    """ringattn_rank_work (host only): per-rank (units, pairs, tiles) as int64 arrays."""
    u = np.zeros(c, dtype=np.int64)
    p = np.zeros(c, dtype=np.int64)
    t = np.zeros(c, dtype=np.int64)
    _check("ringattn_rank_work", lib().ringattn_rank_work(
        S, c, int(causal), layout, tile, u.ctypes.data_as(ctypes.c_void_p),
        p.ctypes.data_as(ctypes.c_void_p), t.ctypes.data_as(ctypes.c_void_p)))
    return u, p, t


def sync_status(stream=None) -> int:
    """ringattn_sync_status: synchronise, return RA_OK or RA_ERR_TIMEOUT / RA_ERR_CUDA."""
    return lib().ringattn_sync_status(ctypes.c_void_p(_stream(stream)))


def last_timeout():
    """ringattn_last_timeout: (barrier smem address, CTA, thread) of the last timeout."""
    info = (ctypes.c_int * 3)()
    _check("ringattn_last_timeout", lib().ringattn_last_timeout(info))
    return tuple(info)


def selftest_timeout(timeout_ns: int, stream=None) -> None:
    _check("ringattn_selftest_timeout", lib().ringattn_selftest_timeout(
        int(timeout_ns), ctypes.c_void_p(_stream(stream))))


def attention(q, k, v, *, c, causal, layout, kv_block, stream=None):
    """Natural-order convenience call: permute q/k/v to rank-major, run the fused
    kernel, permute out/lse back.  Returns (out fp32 [Hq,S,d], lse fp32 [Hq,S])."""
    Hq, S, d = q.shape
    dev = q.device
    qr, kr, vr = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    permute(q, qr, c=c, layout=layout, inverse=0, stream=stream)
    permute(k, kr, c=c, layout=layout, inverse=0, stream=stream)
    permute(v, vr, c=c, layout=layout, inverse=0, stream=stream)
    o_r = torch.empty((Hq, S, d), dtype=torch.float32, device=dev)
    l_r = torch.empty((Hq, S), dtype=torch.float32, device=dev)
    fwd(qr, kr, vr, o_r, l_r, c=c, causal=causal, layout=layout, kv_block=kv_block, stream=stream)
    out = torch.empty_like(o_r)
    lse = torch.empty_like(l_r)
    permute(o_r, out, c=c, layout=layout, inverse=1, stream=stream)
    permute(l_r, lse, c=c, layout=layout, inverse=1, stream=stream)
    return out, lse


def attention_backward(q, k, v, out, lse, dout, *, c, causal, layout, kv_block, stream=None):
    """Natural-order convenience call for the backward pass (ringattn_bwd_natural: the
    chunk map is applied in the kernels' addressing).  ``out`` and ``lse`` are
    :func:`attention`'s results for q, k, v.  Returns (dq, dk, dv), fp32, natural order."""
    Hq, S, d = q.shape
    Hkv = k.shape[0]
    dev = q.device
    dq = torch.empty((Hq, S, d), dtype=torch.float32, device=dev)
    dk = torch.empty((Hkv, S, d), dtype=torch.float32, device=dev)
    dv = torch.empty_like(dk)
    delta = torch.empty((Hq, S), dtype=torch.float32, device=dev)
    bwd(q, k, v, out, lse, dout, dq, dk, dv, delta, c=c, causal=causal, layout=layout, kv_block=kv_block,
        stream=stream, natural=True)
    return dq, dk, dv
