"""Oracle: plain float64 CPU attention, forward and analytic backward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The GPU library and its
Python binding never import it, and the two share no code.

The arithmetic lives in ``attn_oracle.cpp`` (C++17, float64, std::thread); this
module compiles it with the host C++ compiler on first use and marshals numpy
arrays through ctypes.  Every function here works on float64 numpy arrays in the
layouts below; callers widen bf16/fp32 GPU inputs to float64 first.

Layouts (contiguous):
  fixed length  q, o, do, dq [B, Hq, S, D]; k, v, dk, dv [B, Hkv, S, D]; lse [B, Hq, S]
  variable len  q, o, do, dq [T, Hq, D];    k, v, dk, dv [T, Hkv, D];    lse [Hq, T]

Definitions followed (see attn_oracle.cpp for the passages): standard attention
softmax(Q K^T * scale, mask) V with masked scores at -inf; LSE = m + ln(l) of the
scaled scores; the three gradients by the softmax Jacobian.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


class _Params(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("heads_q", ctypes.c_int32),
        ("heads_kv", ctypes.c_int32),
        ("seqlen", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("cu_seqlens", ctypes.POINTER(ctypes.c_int32)),
        ("n_seqs", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("mask", ctypes.c_int32),
        ("row_ptr", ctypes.POINTER(ctypes.c_int32)),
        ("col_idx", ctypes.POINTER(ctypes.c_int32)),
        ("n_row_blocks", ctypes.c_int32),
        ("n_col_blocks", ctypes.c_int32),
        ("block_q", ctypes.c_int32),
        ("block_k", ctypes.c_int32),
        ("causal_in_block", ctypes.c_int32),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle shared library (host compiler, no GPU needed)."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
        ):
            os.makedirs(_BUILD_DIR, exist_ok=True)
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        dp = ctypes.POINTER(ctypes.c_double)
        pp = ctypes.POINTER(_Params)
        lib.oracle_attn_fwd.argtypes = [pp, dp, dp, dp, dp, dp, ctypes.c_int]
        lib.oracle_attn_fwd_blocked.argtypes = [pp, dp, dp, dp, dp, dp, ctypes.c_int, ctypes.c_int]
        lib.oracle_attn_bwd.argtypes = [pp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
        for f in (lib.oracle_attn_fwd, lib.oracle_attn_fwd_blocked, lib.oracle_attn_bwd):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a


def _dptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _make_params(q, k, scale, causal, block_mask, cu_seqlens):
    """Build the C parameter block; returns (params, keepalive list, varlen flag)."""
    keep = []
    p = _Params()
    varlen = cu_seqlens is not None
    if varlen:
        if q.ndim != 3 or k.ndim != 3:
            raise ValueError("variable length expects q [T, Hq, D] and k [T, Hkv, D]")
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        keep.append(cu)
        T, Hq, D = q.shape
        Hkv = k.shape[1]
        lens = np.diff(cu)
        p.batch = len(cu) - 1
        p.seqlen = int(lens.max()) if len(lens) else 0
        p.cu_seqlens = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        p.n_seqs = len(cu) - 1
        if cu[0] != 0 or cu[-1] != T or np.any(lens < 0):
            raise ValueError("cu_seqlens must start at 0, be non-decreasing and end at T")
    else:
        if q.ndim != 4 or k.ndim != 4:
            raise ValueError("fixed length expects q [B, Hq, S, D] and k [B, Hkv, S, D]")
        B, Hq, S, D = q.shape
        Hkv = k.shape[1]
        p.batch, p.seqlen = B, S
        p.cu_seqlens = ctypes.POINTER(ctypes.c_int32)()
        p.n_seqs = 0
    p.heads_q, p.heads_kv, p.head_dim = Hq, Hkv, D
    if Hkv <= 0 or Hq % Hkv:
        raise ValueError("heads_q must be a multiple of heads_kv")
    p.scale = float(scale)
    p.row_ptr = ctypes.POINTER(ctypes.c_int32)()
    p.col_idx = ctypes.POINTER(ctypes.c_int32)()
    if block_mask is not None:
        rp = np.ascontiguousarray(block_mask["row_ptr"], dtype=np.int32)
        ci = np.ascontiguousarray(block_mask["col_idx"], dtype=np.int32)
        keep += [rp, ci]
        p.mask = 2
        p.row_ptr = rp.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        p.col_idx = ci.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        p.n_row_blocks = len(rp) - 1
        p.n_col_blocks = int(block_mask["n_col_blocks"])
        p.block_q = int(block_mask.get("block_q", 64))
        p.block_k = int(block_mask.get("block_k", 64))
        p.causal_in_block = int(block_mask.get("causal_in_block", 1))
    else:
        p.mask = 1 if causal else 0
    return p, keep, varlen


def attn_fwd(q, k, v, *, scale, causal=False, block_mask=None, cu_seqlens=None, nthreads=0):
    """Plain-definition forward.  Returns (o, lse) as float64 arrays."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    p, keep, varlen = _make_params(q, k, scale, causal, block_mask, cu_seqlens)
    o = np.zeros_like(q)
    if varlen:
        lse = np.zeros((q.shape[1], q.shape[0]), dtype=np.float64)
    else:
        lse = np.zeros(q.shape[:3], dtype=np.float64)
    rc = _load().oracle_attn_fwd(ctypes.byref(p), _dptr(q), _dptr(k), _dptr(v), _dptr(o), _dptr(lse), nthreads)
    if rc:
        raise ValueError("oracle_attn_fwd rejected its arguments")
    return o, lse


def attn_fwd_blocked(q, k, v, *, scale, block, causal=False, block_mask=None, cu_seqlens=None, nthreads=0):
    """Streamed online-softmax forward (key blocks of ``block``).  Returns (o, lse)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    p, keep, varlen = _make_params(q, k, scale, causal, block_mask, cu_seqlens)
    o = np.zeros_like(q)
    if varlen:
        lse = np.zeros((q.shape[1], q.shape[0]), dtype=np.float64)
    else:
        lse = np.zeros(q.shape[:3], dtype=np.float64)
    rc = _load().oracle_attn_fwd_blocked(ctypes.byref(p), _dptr(q), _dptr(k), _dptr(v), _dptr(o), _dptr(lse), int(block), nthreads)
    if rc:
        raise ValueError("oracle_attn_fwd_blocked rejected its arguments")
    return o, lse


def attn_bwd(q, k, v, dout, *, scale, causal=False, block_mask=None, cu_seqlens=None, nthreads=0):
    """Analytic backward.  Returns (dq, dk, dv) as float64 arrays."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    p, keep, varlen = _make_params(q, k, scale, causal, block_mask, cu_seqlens)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rc = _load().oracle_attn_bwd(ctypes.byref(p), _dptr(q), _dptr(k), _dptr(v), _dptr(dout), _dptr(dq), _dptr(dk), _dptr(dv), nthreads)
    if rc:
        raise ValueError("oracle_attn_bwd rejected its arguments")
    return dq, dk, dv
