"""PyTorch-facing binding of ln_residual_fwd (include/gbln.h): fused residual
add + LayerNorm over the rows of a CUDA tensor.

Argument marshalling only; the computation runs in libgbattn.so.  There is no
CPU path: a tensor that is not on a CUDA device raises.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import ATTN_BF16, ATTN_F32, LnParamsC, check


def layernorm_residual(x, residual=None, gamma=None, beta=None, *, eps: float = 1e-5, return_sum: bool = True,
                       return_stats: bool = False, stream=None):
    """y = LayerNorm(x + residual) * gamma + beta over the last dimension.

    x, residual: bf16 or float32 CUDA tensors of the same shape [..., cols]
    (made contiguous); gamma, beta: float32 [cols] or None (1 and 0).
    Returns y, plus h = x + residual if ``return_sum`` and (mean, rstd) per row
    (float32) if ``return_stats``.
    """
    lib = _lib.load()
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("x must be bfloat16 or float32")
    cols = x.shape[-1]
    x2 = x.contiguous().reshape(-1, cols)
    r2 = None
    if residual is not None:
        if residual.shape != x.shape or residual.dtype != x.dtype:
            raise ValueError("residual must match x in shape and dtype")
        r2 = residual.contiguous().reshape(-1, cols)
    for name, t in (("gamma", gamma), ("beta", beta)):
        if t is not None and (t.dtype != torch.float32 or t.numel() != cols or not t.is_cuda):
            raise ValueError(f"{name} must be a float32 CUDA tensor of {cols} elements")
    g = gamma.contiguous() if gamma is not None else None
    b = beta.contiguous() if beta is not None else None
    rows = x2.shape[0]
    y = torch.empty_like(x2)
    h = torch.empty_like(x2) if return_sum else None
    mean = torch.empty(rows, dtype=torch.float32, device=x.device) if return_stats else None
    rstd = torch.empty(rows, dtype=torch.float32, device=x.device) if return_stats else None
    p = LnParamsC()
    p.rows, p.cols = rows, cols
    p.x_stride = p.r_stride = p.y_stride = p.h_stride = cols
    p.eps = float(eps)
    p.dtype = ATTN_BF16 if x.dtype == torch.bfloat16 else ATTN_F32
    ptr = lambda t: None if t is None else t.data_ptr()
    st = stream if stream is not None else torch.cuda.current_stream(x.device)
    check(lib.ln_residual_fwd(ctypes.byref(p), ptr(x2), ptr(r2), ptr(g), ptr(b), ptr(y), ptr(h), ptr(mean),
                              ptr(rstd), ctypes.c_void_p(st.cuda_stream)), "ln_residual_fwd")
    out = [y.reshape(x.shape)]
    if return_sum:
        out.append(h.reshape(x.shape))
    if return_stats:
        out += [mean, rstd]
    return out[0] if len(out) == 1 else tuple(out)
