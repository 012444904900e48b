"""Guard regions: the kernels write nothing outside their outputs and workspace.

compute-sanitizer is not available to these tests, so every output tensor and
each workspace is placed inside a larger buffer whose head and tail (4 KiB each)
hold a byte pattern; after the forward and backward calls through the C ABI the
pattern must be intact, and the results must equal those of the same calls
through the binding (which allocates exact-size buffers): O, LSE, dK and dV bit
for bit, dQ within one bf16 unit in the last place (its float32 sum order
varies from run to run).  The workspace is passed with exactly the size the
library asks for, so a write past it would land in the tail guard.

Cases: fixed length with 128-row and 256-row forward units, causal GQA at head
dim 64, a block-sparse mask, packed variable-length sequences, head dim 256,
float32 I/O and the deterministic backward.
"""

import ctypes

import numpy as np
import pytest
import torch

from bwd_flashattention_fwd_sm_gb300 import BlockMask, SeqLens, _lib, attn_bwd, attn_fwd, make_params
from bwd_flashattention_fwd_sm_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


class Guarded:
    """A tensor of `shape` inside a byte buffer with GUARD bytes of PATTERN on each side."""

    def __init__(self, shape, dtype, nbytes=None):
        esz = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape))
        self.nbytes = nbytes if nbytes is not None else n * esz
        body = (self.nbytes + 255) // 256 * 256
        self.buf = torch.full((body + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.buf[GUARD:GUARD + n * esz].view(dtype).view(shape) if n else None
        self.raw = self.buf[GUARD:GUARD + max(self.nbytes, 1)]

    def intact(self):
        head = self.buf[:GUARD]
        tail = self.buf[GUARD + self.nbytes:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


def _case(kind):
    if kind == "pair_units":  # few units: 128-row forward units
        wl = W.Workload("g_pair", 2, 4, 4, 300, 128, "bf16", "none", seed=91)
        return wl, W.make_inputs(wl), {}
    if kind == "full_units":  # 512 units of 256 rows
        wl = W.Workload("g_full", 2, 16, 16, 4096, 128, "bf16", "causal", seed=92)
        return wl, W.make_inputs(wl), {"causal": True}
    if kind == "gqa_d64":
        wl = W.Workload("g_gqa", 1, 8, 2, 520, 64, "bf16", "causal", seed=93)
        return wl, W.make_inputs(wl), {"causal": True}
    if kind == "block":
        wl = W.Workload("g_block", 1, 4, 2, 700, 128, "bf16", "block", seed=94)
        inp = W.make_inputs(wl.with_(mask="none"))
        nb = (700 + 63) // 64
        t = np.random.default_rng(9).random((nb, nb)) < 0.4
        np.fill_diagonal(t, True)
        inp["block_mask"] = W.csr_from_dense_blocks(t)
        return wl, inp, {"block_mask": BlockMask.from_csr(inp["block_mask"], device="cuda")}
    if kind == "varlen":
        lens = [300, 0, 1, 517, 128, 64]
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T = int(cu[-1])
        wl = W.Workload("g_varlen", 1, 4, 2, max(lens), 128, "bf16", "causal", varlen=True, n_seqs=len(lens), seed=95)
        g = torch.Generator().manual_seed(95)
        inp = {n: torch.randn(s, generator=g).to(torch.bfloat16) for n, s in
               (("q", (T, 4, 128)), ("k", (T, 2, 128)), ("v", (T, 2, 128)), ("do", (T, 4, 128)))}
        return wl, inp, {"causal": True, "seqlens": SeqLens(cu, device="cuda"), "seqlen": max(lens)}
    if kind == "d256":
        wl = W.Workload("g_d256", 1, 2, 1, 333, 256, "bf16", "causal", seed=96)
        return wl, W.make_inputs(wl), {"causal": True}
    if kind == "f32":
        wl = W.Workload("g_f32", 1, 2, 2, 130, 128, "f32", "none", seed=97)
        return wl, W.make_inputs(wl), {}
    raise ValueError(kind)


def _lse_shape(q, kw):
    return (q.shape[1], q.shape[0]) if "seqlens" in kw else tuple(q.shape[:3])


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic_dq", "deterministic"])
@pytest.mark.parametrize("kind", ["pair_units", "full_units", "gqa_d64", "block", "varlen", "d256", "f32"])
def test_outputs_and_workspace_guards_intact(kind, deterministic):
    if deterministic and kind in ("d256", "f32"):
        pytest.skip("the deterministic backward runs on the tensor-core path at head dims 64 and 128 only")
    torch.cuda.set_device(0)
    lib = _lib.load()
    wl, inp, kw = _case(kind)
    q, k, v, do = (inp[n].cuda().contiguous() for n in ("q", "k", "v", "do"))
    p = make_params(q, k, scale=wl.scale, **kw)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    o = Guarded(q.shape, q.dtype)
    lse = Guarded(_lse_shape(q, kw), torch.float32)
    wsf = Guarded((0,), torch.uint8, nbytes=lib.attn_fwd_workspace_size(ctypes.byref(p)))
    rc = lib.attn_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o.t), _ptr(lse.t), _ptr(wsf.raw),
                      ctypes.c_size_t(wsf.nbytes), stream)
    assert rc == _lib.ATTN_OK, lib.attn_last_error()

    dq, dk, dv = Guarded(q.shape, q.dtype), Guarded(k.shape, k.dtype), Guarded(v.shape, v.dtype)
    wsb = Guarded((0,), torch.uint8, nbytes=lib.attn_bwd_workspace_size(ctypes.byref(p)))
    fn = lib.attn_bwd_deterministic if deterministic else lib.attn_bwd
    rc = fn(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o.t), _ptr(do), _ptr(lse.t), _ptr(dq.t), _ptr(dk.t),
            _ptr(dv.t), _ptr(wsb.raw), ctypes.c_size_t(wsb.nbytes), stream)
    assert rc == _lib.ATTN_OK, lib.attn_last_error()
    torch.cuda.synchronize()
    assert lib.attn_get_status(None) == _lib.ATTN_OK

    for name, g in (("o", o), ("lse", lse), ("forward workspace", wsf), ("dq", dq), ("dk", dk), ("dv", dv),
                    ("backward workspace", wsb)):
        assert g.intact(), f"{name}[{wl.name}]: bytes outside it were written"

    ro, rl = attn_fwd(q, k, v, scale=wl.scale, **kw)
    rq, rk, rv = attn_bwd(q, k, v, ro, do, rl, scale=wl.scale, deterministic=deterministic, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o.t, ro) and torch.equal(lse.t, rl), f"forward[{wl.name}] differs from the binding's"
    assert torch.equal(dk.t, rk) and torch.equal(dv.t, rv), f"dK, dV[{wl.name}] differ from the binding's"
    if deterministic or wl.dtype == "f32":
        diff_ok = torch.equal(dq.t, rq) if deterministic else bool(
            ((dq.t.float() - rq.float()).abs() <= 1e-5 * (1 + rq.float().abs())).all())
        assert diff_ok, f"dQ[{wl.name}] differs from the binding's"
    else:
        a, b = dq.t.double().cpu().numpy(), rq.double().cpu().numpy()
        _, e = np.frexp(np.maximum(np.abs(a), np.abs(b)))
        ulp = np.ldexp(1.0, e - 8)  # one bf16 unit in the last place of the larger
        assert np.all(np.abs(a - b) <= ulp + 1e-6), f"dQ[{wl.name}] differs from the binding's by more than one bf16 ulp"
