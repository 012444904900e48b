"""GPU parity at head dim 256 against the float64 oracle.

bf16 runs both passes on the tensor cores.  The forward takes one 128-row query
tile per unit, with two S buffers and a 256-column O in tensor memory.  The
backward takes each 128-key tile twice, once per half of the head dim for dK,
dV and dQ, in 64-row query steps.  float32 I/O runs both passes on the float32
kernels.  Tolerances are those of every other test (parity_util).
"""

import numpy as np
import pytest
import torch

from bwd_flashattention_fwd_sm_gb300 import workloads as W

from parity_util import check_all, gpu_run, oracle_run
from test_gpu_parity import small, tiles_csr

pytestmark = pytest.mark.gpu

SHAPES_256 = [(1, 2, 2, 1), (1, 2, 1, 17), (2, 2, 2, 129), (1, 4, 1, 300), (1, 2, 2, 513)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("mask", ["none", "causal", "block"])
@pytest.mark.parametrize("shape", SHAPES_256, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes_d256(shape, mask, dtype):
    B, Hq, Hkv, S = shape
    wl = small(f"d256_{mask}_{dtype}", B, Hq, Hkv, S, 256, dtype, mask, seed=600 + S)
    inp = W.make_inputs(wl.with_(mask="none"))
    if mask == "block":
        inp["block_mask"] = tiles_csr(S, seed=S + 11)
    check_all(wl, gpu_run(wl, inp), oracle_run(wl, inp))


def test_block_mask_empty_row_d256():
    wl = small("d256_empty_row", 1, 2, 1, 384, 256, "bf16", "block", seed=61)
    inp = W.make_inputs(wl.with_(mask="none"))
    inp["block_mask"] = tiles_csr(384, seed=12, empty_row=3)
    got = gpu_run(wl, inp)
    assert np.all(np.isneginf(got["lse"][:, :, 192:256])) and np.all(got["o"][:, :, 192:256] == 0)
    check_all(wl, got, oracle_run(wl, inp))


def test_causal_gqa_s2048_d256():
    """S = 2048, four query heads on one KV head, causal: forward and backward in full."""
    wl = W.Workload("d256_causal_s2048", 1, 4, 1, 2048, 256, "bf16", "causal", seed=62)
    inp = W.make_inputs(wl)
    check_all(wl, gpu_run(wl, inp), oracle_run(wl, inp))


@pytest.mark.parametrize("mask,b,h", [("none", 1, 3), ("causal", 0, 9)])
def test_forward_full_size_sampled_head_d256(mask, b, h):
    """B = 2, H = 16, S = 8192, D = 256: the whole forward on the GPU, one head
    against the oracle."""
    wl = W.Workload("d256_s8192", 2, 16, 16, 8192, 256, "bf16", mask, seed=63)
    inp = W.make_inputs(wl)
    got = gpu_run(wl, inp, passes="fwd")
    one = {n: inp[n][b:b + 1, h:h + 1] for n in ("q", "k", "v", "do")}
    ref = oracle_run(wl.with_(batch=1, heads_q=1, heads_kv=1), one, passes="fwd")
    sub = {n: got[n][b:b + 1, h:h + 1] for n in ("o", "lse")}
    check_all(wl, sub, ref, names=("o", "lse"))


@pytest.mark.parametrize("mask,b,h", [("none", 1, 5), ("causal", 0, 12)])
def test_backward_full_size_sampled_head_d256(mask, b, h):
    """B = 2, H = 16, S = 8192, D = 256 (the benchmarked step): forward and
    backward of every head on the GPU, one head's O, LSE, dQ, dK and dV
    against the oracle."""
    wl = W.Workload("d256_s8192_bwd", 2, 16, 16, 8192, 256, "bf16", mask, seed=65)
    inp = W.make_inputs(wl)
    got = gpu_run(wl, inp)
    one = {n: inp[n][b:b + 1, h:h + 1] for n in ("q", "k", "v", "do")}
    ref = oracle_run(wl.with_(batch=1, heads_q=1, heads_kv=1), one)
    sub = {n: got[n][b:b + 1, h:h + 1] for n in ("o", "lse", "dq", "dk", "dv")}
    check_all(wl, sub, ref)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_d256(causal, dtype):
    """Packed sequences (one empty, ragged lengths) at head dim 256."""
    lens = [5, 0, 129, 1, 300]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    wl = W.Workload("varlen_d256", 1, 4, 2, max(lens), 256, dtype, "causal" if causal else "none",
                    varlen=True, n_seqs=len(lens), seed=64)
    T = int(cu[-1])
    g = torch.Generator().manual_seed(64)
    dt = W.torch_dtype(wl)
    inp = {n: torch.randn(s, generator=g).to(dt) for n, s in
           (("q", (T, 4, 256)), ("k", (T, 2, 256)), ("v", (T, 2, 256)), ("do", (T, 4, 256)))}
    inp["cu_seqlens"] = cu
    check_all(wl, gpu_run(wl, inp), oracle_run(wl, inp, cu=cu))
