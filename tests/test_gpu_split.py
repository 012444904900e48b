"""GPU parity of the forward with a split key range.

With fewer forward units than a GPU has SMs, each unit's key tiles are cut into
2-4 parts, each part writes its unnormalised O, row max and row sum, and a
combine kernel merges them into O and LSE.  These shapes take that path (few
heads, long sequences); the workspace size confirms it (it holds the parts'
partial results).  The backward runs on the forward's O and LSE.  Tolerances
are those of every other test (parity_util).
"""

import ctypes

import numpy as np
import pytest
import torch

from bwd_flashattention_fwd_sm_gb300 import _lib, attn_fwd_fp8, make_params, quantize_fp8
from bwd_flashattention_fwd_sm_gb300 import workloads as W

from parity_util import check_all, gpu_run, oracle_run

pytestmark = pytest.mark.gpu


def _assert_split(wl):
    """The forward workspace holds at least two parts' float32 O for every row."""
    q = torch.empty(W.tensor_shapes(wl)[0], dtype=torch.bfloat16, device="cuda")
    k = torch.empty(W.tensor_shapes(wl)[1], dtype=torch.bfloat16, device="cuda")
    p = make_params(q, k, causal=wl.mask == "causal")
    ws = _lib.load().attn_fwd_workspace_size(ctypes.byref(p))
    rows = wl.batch * wl.heads_q * wl.seqlen
    assert ws >= 2 * rows * wl.head_dim * 4, ws


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mask", ["none", "causal"])
@pytest.mark.parametrize("shape", [(1, 2, 2, 4096), (1, 2, 1, 4200)], ids=lambda s: "x".join(map(str, s)))
def test_split_forward(shape, mask, D):
    B, Hq, Hkv, S = shape
    wl = W.Workload(f"split_{mask}_{D}", B, Hq, Hkv, S, D, "bf16", mask, seed=80 + S)
    _assert_split(wl)
    inp = W.make_inputs(wl)
    check_all(wl, gpu_run(wl, inp), oracle_run(wl, inp))


def test_split_forward_fp8():
    """The FP8 forward's parts carry O times the V reference scale; LSE as every FP8 test."""
    from test_gpu_fp8 import _check_fwd, _inputs
    q, k, v = _inputs(1, 2, 1, 4096, seed=90)
    wl = W.Workload("split_fp8", 1, 2, 1, 4096, 128, "bf16", "causal", seed=90)
    _assert_split(wl)
    f = quantize_fp8(q.cuda(), k.cuda(), v.cuda())
    o, lse = attn_fwd_fp8(f, causal=True, scale=1.0 / np.sqrt(128))
    torch.cuda.synchronize()
    _check_fwd(o, lse, q, k, v, scale=1.0 / np.sqrt(128), causal=True)
