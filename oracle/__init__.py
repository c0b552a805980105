"""fp64 CPU oracle for exact attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
CUDA library never calls it, and it imports nothing from the CUDA library: the
two sides share only the seeded input generators in ``workloads.py``.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over rows);
this module compiles it on demand with gcc and marshals numpy arrays.  Every
function takes and returns float64 arrays in the layouts documented there:

    dense : q,o [B,Sq,Hq,d]  k,v [B,Skv,Hkv,d]  lse [B,Hq,Sq]
    varlen: q,o [Tq,Hq,d]    k,v [Tk,Hkv,d]     lse [Hq,Tq]
    decode: q,o [B,Hq,d]     k,v [B,Lmax,Hkv,d] lse [B,Hq]

Parity status: every function here is pinned by tests/test_oracle_pins.py
(worked examples printed on the pages, closed forms, invariants, brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_SO = os.path.join(_HERE, "libattn_oracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/libattn_oracle.so (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fvisibility=hidden",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, d = ctypes.c_int, ctypes.c_double
            lib.oracle_attn_fwd.argtypes = [_D, _D, _D, _D, _D, i, i, i, i, i, i, d, i, i, i, _I, i,
                                            _D]
            lib.oracle_attn_fwd_varlen.argtypes = [_D, _D, _D, _D, _D, _I, _I, i, i, i, i, d, i, i, i,
                                                   _D]
            lib.oracle_attn_decode.argtypes = [_D, _D, _D, _I, _D, _D, i, i, i, i, i, d, _D]
            lib.oracle_attn_fwd_blockwise.argtypes = [_D, _D, _D, _D, _D, i, i, i, i, i, i, d, i, i,
                                                      i, i, _D, _D]
            lib.oracle_decode_split.argtypes = [_D, _D, _D, _I, _D, _D, i, i, i, i, i, d, i, i]
            lib.oracle_combine.argtypes = [_D, _D, _D, _D, ctypes.c_long, i, i, _D]
            lib.oracle_attn_bwd.argtypes = [_D, _D, _D, _D, _D, _D, _D, i, i, i, i, i, i, d, i, i, i,
                                            _D, _D]
            lib.oracle_num_threads.argtypes = []
            lib.oracle_set_num_threads.argtypes = [i]
            for f in ("oracle_attn_fwd", "oracle_attn_fwd_varlen", "oracle_attn_decode",
                      "oracle_attn_fwd_blockwise", "oracle_decode_split", "oracle_combine",
                      "oracle_attn_bwd", "oracle_num_threads", "oracle_set_num_threads"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _pd(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _pi(a: np.ndarray):
    return a.ctypes.data_as(_I)


def _sink(sink, n: int, what: str):
    """(array or None, pointer or None) for an optional logit-sink vector of n values."""
    if sink is None:
        return None, None
    a = _f64(sink).reshape(-1)
    if a.size != n:
        raise ValueError(f"{what}: sink has {a.size} values, {n} expected")
    return a, _pd(a)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> int:
    """Threads later oracle calls use (timing only; results do not depend on
    it).  Returns the previous count."""
    return int(_load().oracle_set_num_threads(int(n)))


def attn_fwd(q, k, v, scale, causal=False, window=0, n_sink=0, rows=None, sink=None):
    """Dense forward; returns (o [B,R,Hq,d], lse [B,Hq,R]) with R = Sq or len(rows).
    sink: optional logit sink per query head [Hq] (-inf: none)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, Hq, d = q.shape
    _, Skv, Hkv, _ = k.shape
    if rows is None:
        rows_arr, n_rows, prow = None, Sq, None
    else:
        rows_arr = _i32(rows)
        n_rows, prow = int(rows_arr.size), _pi(rows_arr)
    o = np.empty((B, n_rows, Hq, d), np.float64)
    lse = np.empty((B, Hq, n_rows), np.float64)
    sk, psk = _sink(sink, Hq, "attn_fwd")
    rc = _load().oracle_attn_fwd(_pd(q), _pd(k), _pd(v), _pd(o), _pd(lse), B, Hq, Hkv, Sq, Skv, d,
                                 float(scale), int(bool(causal)), int(window), int(n_sink), prow,
                                 n_rows, psk)
    _check(rc, "attn_fwd")
    return o, lse


def attn_fwd_varlen(q, k, v, cu_q, cu_k, scale, causal=False, window=0, n_sink=0, sink=None):
    """Packed forward; returns (o [Tq,Hq,d], lse [Hq,Tq]).  sink: as in attn_fwd."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu_q, cu_k = _i32(cu_q), _i32(cu_k)
    Tq, Hq, d = q.shape
    Hkv = k.shape[1]
    o = np.empty((Tq, Hq, d), np.float64)
    lse = np.empty((Hq, Tq), np.float64)
    sk, psk = _sink(sink, Hq, "attn_fwd_varlen")
    rc = _load().oracle_attn_fwd_varlen(_pd(q), _pd(k), _pd(v), _pd(o), _pd(lse), _pi(cu_q),
                                        _pi(cu_k), int(cu_q.size - 1), Hq, Hkv, d, float(scale),
                                        int(bool(causal)), int(window), int(n_sink), psk)
    _check(rc, "attn_fwd_varlen")
    return o, lse


def attn_decode(q, k, v, seqlens, scale, sink=None):
    """Decode over contiguous caches k,v [B,Lmax,Hkv,d]; returns (o [B,Hq,d], lse [B,Hq]).
    sink: as in attn_fwd."""
    q, k, v, seqlens = _f64(q), _f64(k), _f64(v), _i32(seqlens)
    B, Hq, d = q.shape
    _, Lmax, Hkv, _ = k.shape
    o = np.empty((B, Hq, d), np.float64)
    lse = np.empty((B, Hq), np.float64)
    sk, psk = _sink(sink, Hq, "attn_decode")
    rc = _load().oracle_attn_decode(_pd(q), _pd(k), _pd(v), _pi(seqlens), _pd(o), _pd(lse), B, Hq,
                                    Hkv, d, Lmax, float(scale), psk)
    _check(rc, "attn_decode")
    return o, lse


def attn_fwd_blockwise(q, k, v, scale, causal=False, window=0, n_sink=0, block=128, trace=False,
                       sink=None):
    """Online-softmax forward in key blocks; returns (o, lse[, trace [nblk, 2+d]]).
    sink: as in attn_fwd, applied after the last block."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, Hq, d = q.shape
    _, Skv, Hkv, _ = k.shape
    o = np.empty((B, Sq, Hq, d), np.float64)
    lse = np.empty((B, Hq, Sq), np.float64)
    nblk = (Skv + block - 1) // block
    tr = np.full((max(nblk, 1), 2 + d), np.nan) if trace else None
    sk, psk = _sink(sink, Hq, "attn_fwd_blockwise")
    rc = _load().oracle_attn_fwd_blockwise(_pd(q), _pd(k), _pd(v), _pd(o), _pd(lse), B, Hq, Hkv,
                                           Sq, Skv, d, float(scale), int(bool(causal)), int(window),
                                           int(n_sink), int(block),
                                           _pd(tr) if trace else None, psk)
    _check(rc, "attn_fwd_blockwise")
    return (o, lse, tr[:nblk]) if trace else (o, lse)


def decode_split(q, k, v, seqlens, scale, num_splits, page=16):
    """Per-split partials; returns (o_part [B,Hq,S,d], lse_part [B,Hq,S])."""
    q, k, v, seqlens = _f64(q), _f64(k), _f64(v), _i32(seqlens)
    B, Hq, d = q.shape
    _, Lmax, Hkv, _ = k.shape
    o_part = np.empty((B, Hq, num_splits, d), np.float64)
    lse_part = np.empty((B, Hq, num_splits), np.float64)
    rc = _load().oracle_decode_split(_pd(q), _pd(k), _pd(v), _pi(seqlens), _pd(o_part),
                                     _pd(lse_part), B, Hq, Hkv, d, Lmax, float(scale),
                                     int(num_splits), int(page))
    _check(rc, "decode_split")
    return o_part, lse_part


def combine(o_part, lse_part, sink=None):
    """LSE merge over the split axis (second to last of o_part, last of lse_part).
    sink: optional logit sink per merged row (shape of lse_part without its last axis)."""
    o_part, lse_part = _f64(o_part), _f64(lse_part)
    *lead, S, d = o_part.shape
    rows = int(np.prod(lead)) if lead else 1
    o = np.empty((rows, d), np.float64)
    lse = np.empty((rows,), np.float64)
    sk, psk = _sink(sink, rows, "combine")
    rc = _load().oracle_combine(_pd(o_part), _pd(lse_part), _pd(o), _pd(lse), rows, S, d, psk)
    _check(rc, "combine")
    return o.reshape(*lead, d), lse.reshape(*lead)


def attn_bwd(q, k, v, dout, scale, causal=False, window=0, n_sink=0, sink=None):
    """Gradients of the dense forward for output gradient dout [B,Sq,Hq,d];
    returns (dq [B,Sq,Hq,d], dk [B,Skv,Hkv,d], dv [B,Skv,Hkv,d]), and with a
    logit sink per query head (sink [Hq]) also dsink [Hq]."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Sq, Hq, d = q.shape
    _, Skv, Hkv, _ = k.shape
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    sk, psk = _sink(sink, Hq, "attn_bwd")
    dsink = np.zeros(Hq, np.float64) if sink is not None else None
    rc = _load().oracle_attn_bwd(_pd(q), _pd(k), _pd(v), _pd(dout), _pd(dq), _pd(dk), _pd(dv), B,
                                 Hq, Hkv, Sq, Skv, d, float(scale), int(bool(causal)), int(window),
                                 int(n_sink), psk, None if dsink is None else _pd(dsink))
    _check(rc, "attn_bwd")
    if sink is None:
        return dq, dk, dv
    return dq, dk, dv, dsink
