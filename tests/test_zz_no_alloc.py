"""attn_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Some callers may not call cudaMalloc at all: engines that fix their device
memory budget at start-up and forbid any later allocation, and plug-ins inside
a host framework that owns the device allocator and shares none of it.  They
cannot pass a workspace, so this entry point uses a fixed scratch array inside
the library instead.

These tests call it through the C ABI and compare it with attn_bwd (which gets a
caller-provided workspace) on two calls in a row:
  dK, dV  bit for bit: both come from the same kernels in the same order and
          take no atomics;
  dQ      within the bf16 parity bound of attn_bwd's dQ (its float32 sum order
          varies from run to run) and of the float64 oracle.
The calls cover every part of the shared array: a block-sparse call (its
transposed mask lives there) follows a call with another mask and shape, and a
packed variable-length call (a different work-list size) follows that.  Each
parametrised run starts from a different case, so every case also runs after
another one has left its contents in the array.  A problem too large for the
array is refused before any work, after the same argument checks as attn_bwd.

The file name makes pytest collect it after every other test file.
"""

import ctypes

import numpy as np
import pytest
import torch

from bwd_flashattention_fwd_sm_gb300 import BlockMask, SeqLens, _lib, attn_bwd, attn_fwd, make_params
from bwd_flashattention_fwd_sm_gb300 import workloads as W

from parity_util import compare, oracle_run

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _block_csr(S, seed):
    nb = (S + 63) // 64
    t = np.random.default_rng(seed).random((nb, nb)) < 0.4
    np.fill_diagonal(t, True)
    t &= np.tril(np.ones((nb, nb), bool))
    return W.csr_from_dense_blocks(t, causal_in_block=1)


def _case(kind):
    """Inputs and keyword arguments of one backward problem."""
    if kind == "causal_gqa":
        wl = W.Workload("na_causal_gqa", 1, 8, 2, 1000, 128, "bf16", "causal", seed=21)
        return wl, W.make_inputs(wl), {"causal": True}, None
    if kind == "block":
        wl = W.Workload("na_block", 2, 4, 2, 700, 128, "bf16", "block", seed=22)
        inp = W.make_inputs(wl.with_(mask="none"))
        inp["block_mask"] = _block_csr(700, seed=7)
        return wl, inp, {"block_mask": BlockMask.from_csr(inp["block_mask"], device="cuda")}, None
    if kind == "varlen":
        lens = [300, 0, 1, 517, 128, 64]
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T = int(cu[-1])
        wl = W.Workload("na_varlen", 1, 4, 4, max(lens), 64, "bf16", "causal", varlen=True, n_seqs=len(lens),
                        seed=23)
        g = torch.Generator().manual_seed(23)
        inp = {n: torch.randn(s, generator=g).to(torch.bfloat16) for n, s in
               (("q", (T, 4, 64)), ("k", (T, 4, 64)), ("v", (T, 4, 64)), ("do", (T, 4, 64)))}
        inp["cu_seqlens"] = cu
        return wl, inp, {"causal": True, "seqlens": SeqLens(cu, device="cuda"), "seqlen": max(lens)}, cu
    raise ValueError(kind)


def _noalloc_bwd(q, k, v, o, do, lse, kw, scale):
    lib = _lib.load()
    p = make_params(q, k, scale=scale, **kw)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.attn_bwd_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                              _ptr(dq), _ptr(dk), _ptr(dv), stream)
    return rc, dq, dk, dv


ORDERS = [("causal_gqa", "block", "varlen"), ("block", "varlen", "causal_gqa"), ("varlen", "causal_gqa", "block")]


@pytest.mark.parametrize("order", ORDERS, ids=lambda o: "-".join(o))
def test_noalloc_matches_workspace_entry_point_on_calls_in_a_row(order):
    torch.cuda.set_device(0)
    for kind in order:  # calls in a row on the one shared array
        wl, inp, kw, cu = _case(kind)
        q, k, v, do = (inp[n].cuda().contiguous() for n in ("q", "k", "v", "do"))
        o, lse = attn_fwd(q, k, v, scale=wl.scale, **kw)
        rc, dq, dk, dv = _noalloc_bwd(q, k, v, o, do, lse, kw, wl.scale)
        assert rc == _lib.ATTN_OK, _lib.load().attn_last_error()
        rq, rk, rv = attn_bwd(q, k, v, o, do, lse, scale=wl.scale, **kw)
        torch.cuda.synchronize()
        assert _lib.load().attn_get_status(None) == _lib.ATTN_OK
        tag = f"{wl.name}, after {order[:order.index(kind)]}"
        assert torch.equal(dk, rk), f"dk[{tag}] differs from attn_bwd's"
        assert torch.equal(dv, rv), f"dv[{tag}] differs from attn_bwd's"
        compare(f"dq[{tag}] vs attn_bwd", dq.double().cpu().numpy(), rq.double().cpu().numpy(), "bf16")
        ref = oracle_run(wl, inp, cu=cu)
        compare(f"dq[{tag}] vs oracle", dq.double().cpu().numpy(), ref["dq"], "bf16")


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
    # the same oversized call with a NULL output gets attn_bwd's argument error first
    rc = lib.attn_bwd_noalloc(ctypes.byref(p), dummy, dummy, dummy, dummy, dummy, dummy, None, dummy, dummy, None)
    assert rc == _lib.ATTN_ERR_INVALID_ARG
