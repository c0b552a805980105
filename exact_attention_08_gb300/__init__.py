"""Exact attention on GB300 (sm_103a): thin Python binding of libattn_gb300.so.

Every function here only marshals arguments (device pointers, sizes, the
current CUDA stream) and calls the C ABI declared in include/attn.h of the
same name; all attention arithmetic runs in the library's CUDA kernels.
PyTorch is used for device memory and streams only.  There is no fallback:
importing this package fails if the library cannot be built or loaded, and a
call fails if the library reports an error.

    o, lse = attn_fwd(q, k, v, causal=True)          # q [B,Sq,Hq,d], k/v [B,Skv,Hkv,d]
    o, lse = attn_fwd_ex(q, k, v, cu_q, cu_k, max_seqlen_q=..., causal=True)
    o, lse = attn_decode_paged(q, k_pages, v_pages, page_table, seqlens, num_splits=8)
    o, lse = attn_fwd_ex_sink(q, k, v, sink_logit, causal=True)   # sink_logit [Hq] fp32
    o, lse = attn_decode_paged_sink(q, k_pages, v_pages, page_table, seqlens, sink_logit)
"""
from __future__ import annotations

import ctypes
import math
import os

from . import _build

__all__ = [
    "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_CUDA", "ATTN_ERR_TIMEOUT",
    "ATTN_ERR_BAD_INPUT", "AttnError", "attn_fwd", "attn_fwd_ex", "attn_fwd_ex_sink",
    "attn_fwd_paged", "attn_fwd_strided", "attn_bwd", "attn_bwd_ex", "attn_bwd_ex_sink",
    "attn_bwd_workspace_size",
    "attn_decode_workspace_size", "attn_decode_paged", "attn_decode_paged_sink", "attn_device_status", "attn_check_wait_timeout", "attn_status_string",
    "attn_last_error", "library_path", "lib",
]

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_BAD_INPUT = 5


def _load() -> ctypes.CDLL:
    path = _build.LIB
    if _build.needs_build():
        try:
            path = _build.build()
        except Exception as e:  # no silent fallback: the package is unusable without it
            raise ImportError(f"exact_attention_08_gb300: cannot build {_build.LIB}: {e}") from e
    if not os.path.exists(path):
        raise ImportError(f"exact_attention_08_gb300: {path} is missing")
    L = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp]
    L.attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, i, i, vp]
    L.attn_fwd_ex_sink.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, i, i,
                                   vp, vp]
    L.attn_fwd_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, i,
                                 i, i, vp, vp]
    i64p = ctypes.POINTER(ctypes.c_longlong)
    L.attn_fwd_strided.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i64p, i64p, i64p, i64p, f,
                                   i, i, i, vp, vp]
    L.attn_bwd_workspace_size.argtypes = [i, i, i]
    L.attn_bwd_workspace_size.restype = sz
    L.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp]
    L.attn_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f,
                              i, i, i, vp, sz, vp]
    L.attn_bwd_ex_sink.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i,
                                   i, f, i, i, i, vp, vp, vp, sz, vp]
    L.attn_decode_workspace_size.argtypes = [i, i, i, i]
    L.attn_decode_workspace_size.restype = sz
    L.attn_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp, sz,
                                    vp]
    L.attn_decode_paged_sink.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp,
                                         vp, sz, vp]
    L.attn_device_status.argtypes = [vp]
    L.attn_check_wait_timeout.argtypes = [i, vp]
    L.attn_status_string.argtypes = [i]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_last_error.argtypes = []
    L.attn_last_error.restype = ctypes.c_char_p
    for fn in ("attn_fwd", "attn_fwd_ex", "attn_fwd_ex_sink", "attn_fwd_paged", "attn_fwd_strided",
               "attn_bwd", "attn_bwd_ex", "attn_bwd_ex_sink",
               "attn_decode_paged",
               "attn_decode_paged_sink", "attn_device_status", "attn_check_wait_timeout"):
        getattr(L, fn).restype = ctypes.c_int
    return L


lib = _load()
library_path = _build.LIB


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = lib.attn_last_error().decode()
        msg = f"{what}: {lib.attn_status_string(status).decode()}"
        super().__init__(msg + (f" ({detail})" if detail else ""))


def attn_status_string(status: int) -> str:
    return lib.attn_status_string(int(status)).decode()


def attn_last_error() -> str:
    return lib.attn_last_error().decode()


def _check(rc: int, what: str) -> None:
    if rc != ATTN_OK:
        raise AttnError(rc, what)


def _torch():
    import torch
    return torch


def _stream(stream):
    if stream is None:
        return _torch().cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t, name, dtype, device=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def attn_fwd(q, k, v, o=None, lse=None, *, causal=False, window=0, scale=None, stream=None,
             want_lse=True):
    """Dense BSHD forward.  q [B,Sq,Hq,d], k/v [B,Skv,Hkv,d] bf16 -> o [B,Sq,Hq,d] bf16,
    lse [B,Hq,Sq] fp32 (None when want_lse is False and lse is not given)."""
    torch = _torch()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, q.device)
    B, Sq, Hq, d = q.shape
    Bk, Skv, Hkv, dk = k.shape
    if Bk != B or dk != d or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q/k/v shapes disagree")
    if o is None:
        o = torch.empty_like(q)
    _need(o, "o", torch.bfloat16, q.device)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Skv, d,
                      scale, int(bool(causal)), int(window), _stream(stream))
    _check(rc, "attn_fwd")
    return o, lse


def attn_fwd_ex(q, k, v, cu_seqlens_q=None, cu_seqlens_k=None, *, max_seqlen_q=None,
                max_seqlen_k=None, o=None, lse=None, causal=False, window=0, n_sink=0, scale=None,
                stream=None, want_lse=True):
    """Forward with sink keys and optional packing.  With cu_seqlens (int32 CUDA
    tensors [nseq+1]): q [Tq,Hq,d], k/v [Tk,Hkv,d], o [Tq,Hq,d], lse [Hq,Tq].
    Without: the dense layout of attn_fwd."""
    return _fwd_ex(q, k, v, cu_seqlens_q, cu_seqlens_k, None, max_seqlen_q, max_seqlen_k, o, lse,
                   causal, window, n_sink, scale, stream, want_lse)


def attn_fwd_ex_sink(q, k, v, sink_logit, cu_seqlens_q=None, cu_seqlens_k=None, *,
                     max_seqlen_q=None, max_seqlen_k=None, o=None, lse=None, causal=False,
                     window=0, n_sink=0, scale=None, stream=None, want_lse=True):
    """attn_fwd_ex with a logit sink per query head: sink_logit fp32 CUDA tensor [Hq]
    (-inf entries: no sink for that head)."""
    return _fwd_ex(q, k, v, cu_seqlens_q, cu_seqlens_k, sink_logit, max_seqlen_q, max_seqlen_k,
                   o, lse, causal, window, n_sink, scale, stream, want_lse)


def _fwd_ex(q, k, v, cu_seqlens_q, cu_seqlens_k, sink_logit, max_seqlen_q, max_seqlen_k, o, lse,
            causal, window, n_sink, scale, stream, want_lse):
    torch = _torch()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, q.device)
    varlen = cu_seqlens_q is not None
    if varlen:
        _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, q.device)
        _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, q.device)
        Tq, Hq, d = q.shape
        Tk, Hkv, _ = k.shape
        nseq = cu_seqlens_q.numel() - 1
        if max_seqlen_q is None or max_seqlen_k is None:
            raise ValueError("max_seqlen_q and max_seqlen_k are required with cu_seqlens")
        B, sq, sk = nseq, int(max_seqlen_q), int(max_seqlen_k)
        lse_shape = (Hq, Tq)
    else:
        B, sq, Hq, d = q.shape
        _, sk, Hkv, _ = k.shape
        Tq = Tk = 0
        lse_shape = (B, Hq, sq)
    if o is None:
        o = torch.empty_like(q)
    _need(o, "o", torch.bfloat16, q.device)
    if lse is None and want_lse:
        lse = torch.empty(*lse_shape, dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if sink_logit is None:
        rc = lib.attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens_q),
                             _ptr(cu_seqlens_k), B, Hq, Hkv, sq, sk, Tq, Tk, d, scale,
                             int(bool(causal)), int(window), int(n_sink), _stream(stream))
        _check(rc, "attn_fwd_ex")
    else:
        _need(sink_logit, "sink_logit", torch.float32, q.device)
        if sink_logit.numel() != Hq:
            raise ValueError(f"sink_logit must hold Hq={Hq} values")
        rc = lib.attn_fwd_ex_sink(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                  _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, Hq, Hkv, sq, sk, Tq,
                                  Tk, d, scale, int(bool(causal)), int(window), int(n_sink),
                                  _ptr(sink_logit), _stream(stream))
        _check(rc, "attn_fwd_ex_sink")
    return o, lse


def attn_fwd_paged(q, k_pages, v_pages, page_table, cu_seqlens_q, seqlens_k, o=None, lse=None, *,
                   max_seqlen_q=None, causal=True, window=0, n_sink=0, sink_logit=None,
                   scale=None, stream=None, want_lse=True):
    """Packed queries q [Tq,Hq,d] bf16 against a paged cache k/v_pages [P,16,Hkv,d];
    page_table [B,maxP] int32, cu_seqlens_q [B+1] int32, seqlens_k [B] int32 ->
    o [Tq,Hq,d] bf16, lse [Hq,Tq] fp32.  Causal alignment is to the end of each
    sequence's keys."""
    torch = _torch()
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _need(k_pages, "k_pages", torch.bfloat16, dev)
    _need(v_pages, "v_pages", torch.bfloat16, dev)
    _need(page_table, "page_table", torch.int32, dev)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, dev)
    _need(seqlens_k, "seqlens_k", torch.int32, dev)
    Tq, Hq, d = q.shape
    P, page, Hkv, dk = k_pages.shape
    if dk != d or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("k_pages/v_pages shapes disagree with q")
    B = seqlens_k.numel()
    if page_table.dim() != 2 or page_table.shape[0] != B or cu_seqlens_q.numel() != B + 1:
        raise ValueError("page_table must be [B, max_pages], cu_seqlens_q [B+1], seqlens_k [B]")
    if max_seqlen_q is None:
        raise ValueError("max_seqlen_q is required")
    if o is None:
        o = torch.empty_like(q)
    _need(o, "o", torch.bfloat16, dev)
    if lse is None and want_lse:
        lse = torch.empty(Hq, Tq, dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    if sink_logit is not None:
        _need(sink_logit, "sink_logit", torch.float32, dev)
        if sink_logit.numel() != Hq:
            raise ValueError(f"sink_logit must hold Hq={Hq} values")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = lib.attn_fwd_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                            _ptr(cu_seqlens_q), _ptr(seqlens_k), _ptr(o), _ptr(lse), B, Hq, Hkv,
                            int(max_seqlen_q), Tq, d, page, page_table.shape[1], P, scale,
                            int(bool(causal)), int(window), int(n_sink), _ptr(sink_logit),
                            _stream(stream))
    _check(rc, "attn_fwd_paged")
    return o, lse


def attn_fwd_strided(q, k, v, o=None, lse=None, *, causal=False, window=0, n_sink=0,
                     sink_logit=None, scale=None, stream=None, want_lse=True):
    """Dense forward on q [B,Sq,Hq,d], k/v [B,Skv,Hkv,d] of any strides with d
    contiguous (a BHSD tensor passed as ``t.transpose(1, 2)``, for instance).
    o defaults to ``empty_like(q)`` (same layout); lse is [B,Hq,Sq] contiguous."""
    torch = _torch()
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16:
            raise ValueError(f"{n} must be a bf16 CUDA tensor")
        if t.dim() != 4 or t.stride(3) != 1:
            raise ValueError(f"{n} must be 4-D with a contiguous last dimension")
    B, Sq, Hq, d = q.shape
    Bk, Skv, Hkv, dk = k.shape
    if Bk != B or dk != d or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q/k/v shapes disagree")
    if o is None:
        o = torch.empty_like(q)
    if o.dtype != torch.bfloat16 or tuple(o.shape) != tuple(q.shape) or o.stride(3) != 1:
        raise ValueError("o must be bf16, shaped like q, with a contiguous last dimension")
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    if sink_logit is not None:
        _need(sink_logit, "sink_logit", torch.float32, dev)
        if sink_logit.numel() != Hq:
            raise ValueError(f"sink_logit must hold Hq={Hq} values")

    def strides(t):
        return (ctypes.c_longlong * 3)(t.stride(0), t.stride(1), t.stride(2))

    sq, sk, sv, so = strides(q), strides(k), strides(v), strides(o)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = lib.attn_fwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Skv,
                              d, sq, sk, sv, so, scale, int(bool(causal)), int(window),
                              int(n_sink), _ptr(sink_logit), _stream(stream))
    _check(rc, "attn_fwd_strided")
    return o, lse


def attn_bwd_workspace_size(B: int, Hq: int, Sq: int) -> int:
    return int(lib.attn_bwd_workspace_size(int(B), int(Hq), int(Sq)))


def attn_bwd(q, k, v, o, lse, dout, dq=None, dk=None, dv=None, *, causal=False, scale=None,
             workspace=None, stream=None):
    """Gradients of attn_fwd: q [B,Sq,Hq,d], k/v [B,Skv,Hkv,d], the forward's o and
    lse [B,Hq,Sq], dout like o (all contiguous, bf16 except lse) -> (dq, dk, dv) bf16."""
    torch = _torch()
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _need(t, n, torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    B, Sq, Hq, d = q.shape
    Bk, Skv, Hkv, dk_ = k.shape
    if Bk != B or dk_ != d or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q/k/v shapes disagree")
    if tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("o and dout must be shaped like q")
    if tuple(lse.shape) != (B, Hq, Sq):
        raise ValueError("lse must be [B, Hq, Sq]")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n, ref in ((dq, "dq", q), (dk, "dk", k), (dv, "dv", v)):
        _need(t, n, torch.bfloat16, dev)
        if tuple(t.shape) != tuple(ref.shape):
            raise ValueError(f"{n} has the wrong shape")
    need = attn_bwd_workspace_size(B, Hq, Sq)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                      _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Skv, d, scale, int(bool(causal)),
                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                      _stream(stream))
    _check(rc, "attn_bwd")
    return dq, dk, dv


def attn_bwd_ex(q, k, v, o, lse, dout, cu_seqlens_q=None, cu_seqlens_k=None, dq=None, dk=None,
                dv=None, *, max_seqlen_q=None, max_seqlen_k=None, causal=False, window=0,
                n_sink=0, scale=None, workspace=None, stream=None):
    """Gradients of attn_fwd_ex (sink keys, sliding window, packed sequences).
    With cu_seqlens (int32 CUDA tensors [nseq+1]): q, o, dout [Tq,Hq,d], k/v
    [Tk,Hkv,d], lse [Hq,Tq]; without: the dense layout of attn_bwd."""
    return _bwd_ex(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, dq, dk, dv, None, None,
                   max_seqlen_q, max_seqlen_k, causal, window, n_sink, scale, workspace, stream)


def attn_bwd_ex_sink(q, k, v, o, lse, dout, sink_logit, cu_seqlens_q=None, cu_seqlens_k=None,
                     dq=None, dk=None, dv=None, dsink=None, *, max_seqlen_q=None,
                     max_seqlen_k=None, causal=False, window=0, n_sink=0, scale=None,
                     workspace=None, stream=None):
    """Gradients of attn_fwd_ex_sink: (dq, dk, dv, dsink), dsink fp32 [Hq]
    the gradient of the logit sink.  lse is the forward's (sink included)."""
    torch = _torch()
    _need(sink_logit, "sink_logit", torch.float32, q.device)
    Hq = q.shape[-2]
    if sink_logit.numel() != Hq:
        raise ValueError(f"sink_logit must hold Hq={Hq} values")
    dsink = torch.empty(Hq, dtype=torch.float32, device=q.device) if dsink is None else dsink
    _need(dsink, "dsink", torch.float32, q.device)
    if dsink.numel() != Hq:
        raise ValueError(f"dsink must hold Hq={Hq} values")
    return _bwd_ex(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, dq, dk, dv,
                   sink_logit.contiguous(), dsink, max_seqlen_q, max_seqlen_k, causal, window,
                   n_sink, scale, workspace, stream)


def _bwd_ex(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, dq, dk, dv, sink_logit, dsink,
            max_seqlen_q, max_seqlen_k, causal, window, n_sink, scale, workspace, stream):
    torch = _torch()
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _need(t, n, torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    varlen = cu_seqlens_q is not None
    if varlen:
        _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, dev)
        _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, dev)
        Tq, Hq, d = q.shape
        Tk, Hkv, dk_ = k.shape
        if max_seqlen_q is None or max_seqlen_k is None:
            raise ValueError("max_seqlen_q and max_seqlen_k are required with cu_seqlens")
        B, sq, sk = cu_seqlens_q.numel() - 1, int(max_seqlen_q), int(max_seqlen_k)
        lse_shape = (Hq, Tq)
    else:
        B, sq, Hq, d = q.shape
        Bk, sk, Hkv, dk_ = k.shape
        if Bk != B:
            raise ValueError("q/k batch sizes disagree")
        Tq = Tk = 0
        lse_shape = (B, Hq, sq)
    if dk_ != d or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q/k/v shapes disagree")
    if tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("o and dout must be shaped like q")
    if tuple(lse.shape) != lse_shape:
        raise ValueError(f"lse must be {list(lse_shape)}")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n, ref in ((dq, "dq", q), (dk, "dk", k), (dv, "dv", v)):
        _need(t, n, torch.bfloat16, dev)
        if tuple(t.shape) != tuple(ref.shape):
            raise ValueError(f"{n} has the wrong shape")
    need = attn_bwd_workspace_size(B, Hq, sq)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
            _ptr(dv), _ptr(cu_seqlens_q) if varlen else None,
            _ptr(cu_seqlens_k) if varlen else None, B, Hq, Hkv, sq, sk, Tq, Tk, d, scale,
            int(bool(causal)), int(window), int(n_sink))
    tail = (_ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if sink_logit is None:
        _check(lib.attn_bwd_ex(*args, *tail), "attn_bwd_ex")
        return dq, dk, dv
    _check(lib.attn_bwd_ex_sink(*args, _ptr(sink_logit), _ptr(dsink), *tail), "attn_bwd_ex_sink")
    return dq, dk, dv, dsink


def attn_decode_workspace_size(B: int, Hq: int, d: int, num_splits: int) -> int:
    return int(lib.attn_decode_workspace_size(int(B), int(Hq), int(d), int(num_splits)))


def attn_decode_paged(q, k_pages, v_pages, page_table, seqlens, o=None, lse=None, *,
                      num_splits=8, scale=None, workspace=None, stream=None, want_lse=True):
    """One-token decode.  q [B,Hq,d] bf16, k/v_pages [P,16,Hkv,d] bf16, page_table
    [B,maxP] int32, seqlens [B] int32 -> o [B,Hq,d] bf16, lse [B,Hq] fp32."""
    return _decode(q, k_pages, v_pages, page_table, seqlens, None, o, lse, num_splits, scale,
                   workspace, stream, want_lse)


def attn_decode_paged_sink(q, k_pages, v_pages, page_table, seqlens, sink_logit, o=None,
                           lse=None, *, num_splits=8, scale=None, workspace=None, stream=None,
                           want_lse=True):
    """attn_decode_paged with a logit sink per query head: sink_logit fp32 CUDA tensor [Hq]."""
    return _decode(q, k_pages, v_pages, page_table, seqlens, sink_logit, o, lse, num_splits,
                   scale, workspace, stream, want_lse)


def _decode(q, k_pages, v_pages, page_table, seqlens, sink_logit, o, lse, num_splits, scale,
            workspace, stream, want_lse):
    torch = _torch()
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _need(k_pages, "k_pages", torch.bfloat16, dev)
    _need(v_pages, "v_pages", torch.bfloat16, dev)
    _need(page_table, "page_table", torch.int32, dev)
    _need(seqlens, "seqlens", torch.int32, dev)
    B, Hq, d = q.shape
    P, page, Hkv, dk = k_pages.shape
    if dk != d or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("k_pages/v_pages shapes disagree with q")
    if page_table.dim() != 2 or page_table.shape[0] != B or seqlens.numel() != B:
        raise ValueError("page_table must be [B, max_pages] and seqlens [B]")
    if o is None:
        o = torch.empty_like(q)
    _need(o, "o", torch.bfloat16, dev)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    need = attn_decode_workspace_size(B, Hq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    wbytes = workspace.numel() * workspace.element_size()
    if sink_logit is None:
        rc = lib.attn_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                   _ptr(seqlens), _ptr(o), _ptr(lse), B, Hq, Hkv, d, page,
                                   page_table.shape[1], P, int(num_splits), scale, _ptr(workspace),
                                   wbytes, _stream(stream))
        _check(rc, "attn_decode_paged")
    else:
        _need(sink_logit, "sink_logit", torch.float32, dev)
        if sink_logit.numel() != Hq:
            raise ValueError(f"sink_logit must hold Hq={Hq} values")
        rc = lib.attn_decode_paged_sink(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                        _ptr(seqlens), _ptr(o), _ptr(lse), B, Hq, Hkv, d, page,
                                        page_table.shape[1], P, int(num_splits), scale,
                                        _ptr(sink_logit), _ptr(workspace), wbytes, _stream(stream))
        _check(rc, "attn_decode_paged_sink")
    return o, lse


def attn_device_status(stream=None) -> int:
    """Synchronises the stream; returns and clears the device status word."""
    return int(lib.attn_device_status(_stream(stream)))


def attn_check_wait_timeout(limit_us: int, stream=None) -> None:
    _check(lib.attn_check_wait_timeout(int(limit_us), _stream(stream)), "attn_check_wait_timeout")
