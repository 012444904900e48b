"""GPU parity for position-major storage: Q, K, V, dO (and O, dQ, dK, dV) held as
[batch, seq, heads, head_dim] and passed through the C ABI by their strides, so
the kernels' TMA maps take the dimension order (head dim, head, position, batch).

The Python binding makes tensors contiguous in [batch, heads, seq, head_dim];
these tests call libgbattn directly to keep the strided layout.  Tolerances are
those of every other test (parity_util).
"""

import ctypes

import numpy as np
import pytest
import torch

from bwd_flashattention_fwd_sm_gb300 import _lib, make_params
from bwd_flashattention_fwd_sm_gb300 import workloads as W

from parity_util import check_all, oracle_run

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _run_strided(inp, causal, scale):
    """Forward and backward on [B, S, H, D] storage; results returned as [B, H, S, D]."""
    lib = _lib.load()
    bshd = {n: inp[n].transpose(1, 2).contiguous().to(DEV) for n in ("q", "k", "v", "do")}
    view = {n: t.transpose(1, 2) for n, t in bshd.items()}  # [B, H, S, D] views, position-major strides
    q, k, v, do = view["q"], view["k"], view["v"], view["do"]
    assert not q.is_contiguous()
    p = make_params(q, k, causal=causal, scale=scale)
    o = torch.empty_like(bshd["q"]).transpose(1, 2)
    dq = torch.empty_like(bshd["q"]).transpose(1, 2)
    dk = torch.empty_like(bshd["k"]).transpose(1, 2)
    dv = torch.empty_like(bshd["v"]).transpose(1, 2)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    wf = lib.attn_fwd_workspace_size(ctypes.byref(p))
    wb = lib.attn_bwd_workspace_size(ctypes.byref(p))
    ws = torch.empty(max(wf, wb, 1), dtype=torch.uint8, device=DEV)
    rc = lib.attn_fwd(ctypes.byref(p), _p(q), _p(k), _p(v), _p(o), _p(lse), _p(ws), ctypes.c_size_t(ws.numel()), st)
    assert rc == _lib.ATTN_OK, lib.attn_last_error()
    rc = lib.attn_bwd(ctypes.byref(p), _p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv), _p(ws),
                      ctypes.c_size_t(ws.numel()), st)
    assert rc == _lib.ATTN_OK, lib.attn_last_error()
    torch.cuda.synchronize()
    assert lib.attn_get_status(st) == _lib.ATTN_OK
    out = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    return {n: t.double().cpu().numpy() for n, t in out.items()}


@pytest.mark.parametrize("D,mask,dtype", [(128, "causal", "bf16"), (64, "none", "bf16"), (256, "causal", "bf16"),
                                          (128, "none", "f32")])
def test_position_major_storage(D, mask, dtype):
    wl = W.Workload(f"bshd_{D}_{mask}_{dtype}", 2, 4, 2, 300, D, dtype, mask, seed=70 + D)
    inp = W.make_inputs(wl)
    got = _run_strided(inp, mask == "causal", wl.scale)
    check_all(wl, got, oracle_run(wl, inp))
