"""PyTorch-facing binding of libgbattn: attn_fwd / attn_bwd over CUDA tensors.

Argument marshalling only.  Every step of the computation runs in the library's
CUDA kernels; PyTorch supplies device memory (outputs and workspace) and the
current stream.  There is no CPU path: if the library cannot load, or a tensor
is not on a CUDA device, the call raises.

Layouts (see include/gbattn.h):
  fixed length     q, do [B, Hq, S, D]; k, v [B, Hkv, S, D]; lse [B, Hq, S] float32
  variable length  q, do [T, Hq, D];    k, v [T, Hkv, D];    lse [Hq, T]   float32
                   with ``seqlens`` (a SeqLens) giving the packed sequence starts.
q-like tensors (q, o, do, dq) are made contiguous, as are the kv-like ones, so
each group shares one stride set as the C ABI requires.
"""

from __future__ import annotations

import ctypes
import math

import numpy as np
import torch

from . import _lib
from ._lib import (ATTN_BF16, ATTN_F32, ATTN_MASK_BLOCK, ATTN_MASK_CAUSAL, ATTN_MASK_NONE,
                   SIZE_MAX, BlockMaskC, ParamsC, check)


class BlockMask:
    """A 64x64-tile block-sparse mask: CSR lists by query block, held on host and device.

    ``row_ptr`` [n_blocks + 1] and ``col_idx`` [nnz] (int32, columns strictly
    ascending in each row).  ``causal_in_block`` = 1 also applies j <= i inside
    listed tiles.  One mask serves every batch entry and head.
    """

    def __init__(self, row_ptr, col_idx, n_blocks: int, causal_in_block: int = 1, device=None, block: int = 64):
        self.row_ptr_host = np.ascontiguousarray(row_ptr, dtype=np.int32)
        self.col_idx_host = np.ascontiguousarray(col_idx, dtype=np.int32)
        if self.col_idx_host.size == 0:
            self.col_idx_host = np.zeros(1, dtype=np.int32)[:0]
        self.n_blocks = int(n_blocks)
        self.causal_in_block = int(causal_in_block)
        self.block = int(block)
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.row_ptr = torch.from_numpy(self.row_ptr_host.copy()).to(dev)
        self.col_idx = torch.from_numpy(np.concatenate([self.col_idx_host, np.zeros(1, np.int32)])).to(dev)
        self._c = BlockMaskC()
        self._c.row_ptr = self.row_ptr.data_ptr()
        self._c.col_idx = self.col_idx.data_ptr()
        self._c.row_ptr_host = self.row_ptr_host.ctypes.data
        self._c.col_idx_host = self.col_idx_host.ctypes.data if self.col_idx_host.size else self.row_ptr_host.ctypes.data
        self._c.block_q = self._c.block_k = self.block
        self._c.n_row_blocks = self._c.n_col_blocks = self.n_blocks
        self._c.nnz = int(self.row_ptr_host[-1])
        self._c.causal_in_block = self.causal_in_block

    @classmethod
    def from_csr(cls, csr: dict, device=None) -> "BlockMask":
        return cls(csr["row_ptr"], csr["col_idx"], csr["n_row_blocks"], csr.get("causal_in_block", 1),
                   device=device, block=csr.get("block_q", 64))


class SeqLens:
    """Packed variable-length batch: sequence starts on host and device."""

    def __init__(self, cu_seqlens, device=None):
        self.host = np.ascontiguousarray(np.asarray(cu_seqlens), dtype=np.int32)
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.device = torch.from_numpy(self.host.copy()).to(dev)
        self.n_seqs = len(self.host) - 1
        self.total = int(self.host[-1])
        self.max_len = int(np.max(np.diff(self.host))) if self.n_seqs > 0 else 0


_DTYPES = {torch.float32: ATTN_F32, torch.bfloat16: ATTN_BF16}


def _stream_handle(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_params(q, k, *, causal=False, block_mask: BlockMask | None = None, scale=None,
                seqlens: SeqLens | None = None, seqlen: int | None = None):
    """Fill the C parameter block from tensor shapes and strides."""
    if not (q.is_cuda and k.is_cuda):
        raise ValueError("gbattn runs on CUDA tensors only")
    if q.dtype not in _DTYPES or k.dtype != q.dtype:
        raise ValueError(f"unsupported dtypes q={q.dtype} k={k.dtype}: float32 or bfloat16, both the same")
    p = ParamsC()
    D = q.shape[-1]
    if seqlens is not None:
        if q.dim() != 3 or k.dim() != 3:
            raise ValueError("variable length expects q [T, Hq, D] and k [T, Hkv, D]")
        if q.shape[0] != seqlens.total or k.shape[0] != seqlens.total:
            raise ValueError("packed tensors must have cu_seqlens[-1] rows")
        p.batch = 0
        p.heads_q, p.heads_kv = q.shape[1], k.shape[1]
        p.seqlen = int(seqlen) if seqlen is not None else seqlens.max_len
        p.cu_seqlens = seqlens.device.data_ptr()
        p.cu_seqlens_host = seqlens.host.ctypes.data
        p.n_seqs = seqlens.n_seqs
        p.q_stride_b, p.q_stride_h, p.q_stride_s = 0, q.stride(1), q.stride(0)
        p.kv_stride_b, p.kv_stride_h, p.kv_stride_s = 0, k.stride(1), k.stride(0)
    else:
        if q.dim() != 4 or k.dim() != 4:
            raise ValueError("fixed length expects q [B, Hq, S, D] and k [B, Hkv, S, D]")
        if q.shape[0] != k.shape[0] or q.shape[2] != k.shape[2] or k.shape[3] != D:
            raise ValueError(f"shape mismatch q={tuple(q.shape)} k={tuple(k.shape)}")
        p.batch, p.heads_q, p.seqlen = q.shape[0], q.shape[1], q.shape[2]
        p.heads_kv = k.shape[1]
        p.cu_seqlens = None
        p.cu_seqlens_host = None
        p.n_seqs = 0
        p.q_stride_b, p.q_stride_h, p.q_stride_s = q.stride(0), q.stride(1), q.stride(2)
        p.kv_stride_b, p.kv_stride_h, p.kv_stride_s = k.stride(0), k.stride(1), k.stride(2)
    p.head_dim = D
    p.scale = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    p.dtype = _DTYPES[q.dtype]
    if block_mask is not None:
        p.mask = ATTN_MASK_BLOCK
        p.block_mask = ctypes.pointer(block_mask._c)
    else:
        p.mask = ATTN_MASK_CAUSAL if causal else ATTN_MASK_NONE
    return p


def _workspace(nbytes: int, device, workspace=None):
    if nbytes == SIZE_MAX:
        raise _lib.AttnError(_lib.ATTN_ERR_INVALID_ARG, "workspace size", _lib.load().attn_last_error().decode())
    if nbytes == 0:
        return None
    if workspace is not None and workspace.numel() * workspace.element_size() >= nbytes:
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def fwd_workspace_size(params: ParamsC) -> int:
    return _lib.load().attn_fwd_workspace_size(ctypes.byref(params))


def bwd_workspace_size(params: ParamsC) -> int:
    return _lib.load().attn_bwd_workspace_size(ctypes.byref(params))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def attn_fwd(q, k, v, *, causal=False, block_mask: BlockMask | None = None, scale=None,
             seqlens: SeqLens | None = None, seqlen: int | None = None, stream=None, workspace=None,
             out=None):
    """O, LSE = attention forward.  Returns (o, lse)."""
    lib = _lib.load()
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    if v.shape != k.shape or v.dtype != k.dtype:
        raise ValueError("v must match k in shape and dtype")
    p = make_params(q, k, causal=causal, block_mask=block_mask, scale=scale, seqlens=seqlens, seqlen=seqlen)
    o = out if out is not None else torch.empty_like(q)
    if seqlens is not None:
        lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    else:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    ws = _workspace(lib.attn_fwd_workspace_size(ctypes.byref(p)), q.device, workspace)
    check(lib.attn_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(ws),
                       ctypes.c_size_t(0 if ws is None else ws.numel()), _stream_handle(stream)), "attn_fwd")
    return o, lse


def attn_bwd(q, k, v, o, do, lse, *, causal=False, block_mask: BlockMask | None = None, scale=None,
             seqlens: SeqLens | None = None, seqlen: int | None = None, stream=None, workspace=None,
             deterministic=False):
    """dQ, dK, dV of the attention forward.  Returns (dq, dk, dv).

    deterministic: bit-identical results from run to run (attn_bwd_deterministic:
    dQ from a query-stationary pass; bf16 only)."""
    lib = _lib.load()
    q, k, v, o, do = (t.contiguous() for t in (q, k, v, o, do))
    lse = lse.contiguous()
    if o.shape != q.shape or do.shape != q.shape or v.shape != k.shape:
        raise ValueError("o and do must match q; v must match k")
    if lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    p = make_params(q, k, causal=causal, block_mask=block_mask, scale=scale, seqlens=seqlens, seqlen=seqlen)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ws = _workspace(lib.attn_bwd_workspace_size(ctypes.byref(p)), q.device, workspace)
    name = "attn_bwd_deterministic" if deterministic else "attn_bwd"
    check(getattr(lib, name)(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                             _ptr(dk), _ptr(dv), _ptr(ws), ctypes.c_size_t(0 if ws is None else ws.numel()),
                             _stream_handle(stream)), name)
    return dq, dk, dv


class Fp8Operands:
    """Per-tile e4m3 codes and scales of Q, K, V (attn_quantize_fp8's outputs).

    q8 [B, Hq, S, 128] and k8 [B, Hkv, S, 128] uint8; v8t [B, Hkv, 128, ld] uint8
    (V's codes transposed, ld = S rounded up to 16); q_scale [B, Hq, n_tiles],
    k_scale and v_scale [B, Hkv, n_tiles] float32 with n_tiles = ceil(S / 128).
    """

    def __init__(self, q8, k8, v8t, q_scale, k_scale, v_scale):
        self.q8, self.k8, self.v8t = q8, k8, v8t
        self.q_scale, self.k_scale, self.v_scale = q_scale, k_scale, v_scale

    @classmethod
    def empty(cls, batch, heads_q, heads_kv, seqlen, device):
        ld = (seqlen + 15) // 16 * 16
        nt = (seqlen + 127) // 128
        u8, f32 = torch.uint8, torch.float32
        return cls(torch.empty((batch, heads_q, seqlen, 128), dtype=u8, device=device),
                   torch.empty((batch, heads_kv, seqlen, 128), dtype=u8, device=device),
                   torch.empty((batch, heads_kv, 128, ld), dtype=u8, device=device),
                   torch.empty((batch, heads_q, nt), dtype=f32, device=device),
                   torch.empty((batch, heads_kv, nt), dtype=f32, device=device),
                   torch.empty((batch, heads_kv, nt), dtype=f32, device=device))


def quantize_fp8(q, k, v, *, stream=None, out: Fp8Operands | None = None) -> Fp8Operands:
    """Per-tile e4m3 quantisation of bf16 q [B, Hq, S, 128], k, v [B, Hkv, S, 128]."""
    lib = _lib.load()
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    if v.shape != k.shape or v.dtype != k.dtype:
        raise ValueError("v must match k in shape and dtype")
    p = make_params(q, k)
    f = out if out is not None else Fp8Operands.empty(q.shape[0], q.shape[1], k.shape[1], q.shape[2], q.device)
    check(lib.attn_quantize_fp8(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(f.q8), _ptr(f.k8), _ptr(f.v8t),
                                _ptr(f.q_scale), _ptr(f.k_scale), _ptr(f.v_scale), _stream_handle(stream)),
          "attn_quantize_fp8")
    return f


def attn_fwd_fp8(f: Fp8Operands, *, causal=False, block_mask: BlockMask | None = None, scale=None, stream=None,
                 workspace=None, out=None):
    """O (bf16), LSE of attention on the dequantised FP8 operands.  Returns (o, lse)."""
    lib = _lib.load()
    B, Hq, S, D = f.q8.shape
    o = out if out is not None else torch.empty((B, Hq, S, D), dtype=torch.bfloat16, device=f.q8.device)
    # the parameter block: q strides describe the bf16 O; K and V are the codes' fixed layouts
    p = make_params(o, o, causal=causal, block_mask=block_mask, scale=scale)
    Hkv = f.k8.shape[1]
    p.heads_kv = Hkv
    p.kv_stride_b, p.kv_stride_h, p.kv_stride_s = Hkv * S * D, S * D, D
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=f.q8.device)
    ws = _workspace(lib.attn_fwd_workspace_size(ctypes.byref(p)), f.q8.device, workspace)
    check(lib.attn_fwd_fp8(ctypes.byref(p), _ptr(f.q8), _ptr(f.k8), _ptr(f.v8t), _ptr(f.q_scale), _ptr(f.k_scale),
                           _ptr(f.v_scale), _ptr(o), _ptr(lse), _ptr(ws),
                           ctypes.c_size_t(0 if ws is None else ws.numel()), _stream_handle(stream)), "attn_fwd_fp8")
    return o, lse


def get_status(stream=None) -> int:
    """Wait for the stream; return and clear the device status word."""
    return _lib.load().attn_get_status(_stream_handle(stream))
