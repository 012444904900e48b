"""attn_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Such callers (code running under CUDA-graph stream capture, engines with a fixed
memory budget, plug-ins inside a framework that owns the allocator) cannot pass a
workspace, so this entry point uses a fixed scratch array inside the library.
These tests call it through the C ABI and check its dQ, dK, dV against attn_bwd
with a caller-provided workspace, on two calls in a row with different problems
(the second must not depend on what the first left in the shared array), and
check that a problem too large for the array is refused before any work.

The file name makes pytest collect it after every other test file.
"""

import ctypes

import numpy as np
import pytest
import torch

from bwd_flashattention_fwd_sm_gb300 import _lib, attn_bwd, attn_fwd, make_params
from bwd_flashattention_fwd_sm_gb300 import workloads as W

from parity_util import compare

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc_bwd(q, k, v, o, do, lse, causal, scale):
    lib = _lib.load()
    p = make_params(q, k, causal=causal, scale=scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.attn_bwd_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                              _ptr(dq), _ptr(dk), _ptr(dv), stream)
    return rc, dq, dk, dv


@pytest.mark.parametrize("call", [0, 1])
def test_noalloc_matches_workspace_entry_point_twice(call):
    torch.cuda.set_device(0)
    cases = [W.Workload("na_causal_gqa", 1, 8, 2, 1000, 128, "bf16", "causal", seed=21),
             W.Workload("na_dense", 2, 4, 4, 640, 128, "bf16", "none", seed=22)]
    results = []
    for wl in cases:  # two calls in a row on the shared array
        inp = W.make_inputs(wl)
        q, k, v, do = (inp[n].cuda().contiguous() for n in ("q", "k", "v", "do"))
        causal = wl.mask == "causal"
        o, lse = attn_fwd(q, k, v, causal=causal, scale=wl.scale)
        rc, dq, dk, dv = _noalloc_bwd(q, k, v, o, do, lse, causal, wl.scale)
        assert rc == _lib.ATTN_OK, _lib.load().attn_last_error()
        rq, rk, rv = attn_bwd(q, k, v, o, do, lse, causal=causal, scale=wl.scale)
        torch.cuda.synchronize()
        assert _lib.load().attn_get_status(None) == _lib.ATTN_OK
        for name, a, b in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            compare(f"{name}[{wl.name}, call {call}]", a.double().cpu().numpy(), b.double().cpu().numpy(), "bf16")
        results.append(dq.float().abs().sum().item())
    assert all(np.isfinite(results))


def test_noalloc_refuses_problems_beyond_its_array():
    lib = _lib.load()
    # 4 x 16 heads x 4096 positions x 128 float32 accumulator alone is 128 MiB > 32 MiB
    q = torch.empty((4, 16, 4096, 128), dtype=torch.bfloat16, device="cuda")
    p = make_params(q, q, causal=True)
    need = lib.attn_bwd_workspace_size(ctypes.byref(p))
    assert need > _lib.NOALLOC_SCRATCH_BYTES
    dummy = _ptr(q)
    rc = lib.attn_bwd_noalloc(ctypes.byref(p), dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                              None)
    assert rc == _lib.ATTN_ERR_WORKSPACE
    assert b"fixed" in lib.attn_last_error()
