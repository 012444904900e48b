"""Calls on two CUDA streams at once.

Each call keeps its state in its own workspace (the work list and the unit
counter the persistent CTAs draw from) and no CTA waits on another CTA, so two
problems queued on two streams without any synchronisation between them, whose
kernels then share the SMs, must give the results they give one after the
other: O, LSE, dK and dV bit for bit, dQ within one bf16 unit in the last place
(its float32 sum order varies from run to run).
"""

import numpy as np
import pytest
import torch

from bwd_flashattention_fwd_sm_gb300 import BlockMask, attn_bwd, attn_fwd
from bwd_flashattention_fwd_sm_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _problem(wl, block=None):
    inp = W.make_inputs(wl.with_(mask="none") if block is not None else wl)
    dev = torch.device("cuda")
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    kw = {"scale": wl.scale}
    if wl.mask == "causal":
        kw["causal"] = True
    if block is not None:
        kw["block_mask"] = BlockMask.from_csr(block, device=dev)
    return q, k, v, do, kw


def _run(q, k, v, do, kw, stream):
    with torch.cuda.stream(stream):
        o, lse = attn_fwd(q, k, v, stream=stream, **kw)
        dq, dk, dv = attn_bwd(q, k, v, o, do, lse, stream=stream, **kw)
    return o, lse, dq, dk, dv


def _close_dq(a, b):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    _, e = np.frexp(np.maximum(np.abs(a), np.abs(b)))
    return bool(np.all(np.abs(a - b) <= np.ldexp(1.0, e - 8) + 1e-6))


def test_two_streams_match_one_after_the_other():
    torch.cuda.set_device(0)
    nb = (1500 + 63) // 64
    t = np.random.default_rng(4).random((nb, nb)) < 0.35
    np.fill_diagonal(t, True)
    problems = [
        _problem(W.Workload("st_causal", 2, 16, 4, 2048, 128, "bf16", "causal", seed=31)),
        _problem(W.Workload("st_block", 1, 8, 8, 1500, 64, "bf16", "block", seed=32), W.csr_from_dense_blocks(t)),
    ]
    s0 = torch.cuda.current_stream()
    ref = [_run(*p, s0) for p in problems]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for rep in range(3):
        got = [_run(*p, s) for p, s in zip(problems, streams)]
        torch.cuda.synchronize()
        for j, (g, r) in enumerate(zip(got, ref)):
            for name, a, b in zip(("o", "lse", "dk", "dv"), (g[0], g[1], g[3], g[4]), (r[0], r[1], r[3], r[4])):
                assert torch.equal(a, b), f"{name} of problem {j} differs on two streams (repeat {rep})"
            assert _close_dq(g[2], r[2]), f"dq of problem {j} differs on two streams (repeat {rep})"
