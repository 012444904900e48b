"""GPU parity of the deterministic backward (attn_bwd_deterministic: dK/dV from
the dK/dV-stationary pass, dQ from a query-stationary pass that sums over key
tiles in a fixed order) against the float64 oracle, and its run-to-run
bit-identity.

The tolerances are those of every other bf16 test (parity_util).  Bit-identity
is checked on whole output tensors of two calls on the same inputs.
"""

import numpy as np
import pytest
import torch

from bwd_flashattention_fwd_sm_gb300 import BlockMask, SeqLens, attn_bwd, attn_fwd, get_status
from bwd_flashattention_fwd_sm_gb300 import workloads as W

from parity_util import check_all, gpu_run, oracle_run
from test_gpu_parity import SMALL_SHAPES, _slice_heads, small, tiles_csr

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mask", ["none", "causal", "block"])
@pytest.mark.parametrize("shape", SMALL_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes_deterministic(shape, mask, D):
    B, Hq, Hkv, S = shape
    wl = small(f"det_{mask}", B, Hq, Hkv, S, D, "bf16", mask, seed=200 + S)
    inp = W.make_inputs(wl.with_(mask="none"))
    if mask == "block":
        inp["block_mask"] = tiles_csr(S, seed=S + 1)
    check_all(wl, gpu_run(wl, inp, deterministic=True), oracle_run(wl, inp))


def test_block_mask_empty_row_block_deterministic():
    """A query block with no listed tile gets dQ = 0 from the query-stationary pass."""
    wl = small("det_empty_row", 1, 2, 2, 384, 128, "bf16", "block", seed=7)
    inp = W.make_inputs(wl.with_(mask="none"))
    inp["block_mask"] = tiles_csr(384, seed=5, empty_row=3)
    got = gpu_run(wl, inp, deterministic=True)
    assert np.all(got["dq"][:, :, 192:256] == 0)
    check_all(wl, got, oracle_run(wl, inp))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_deterministic(causal, D):
    lens = [5, 0, 128, 1, 300, 64, 129, 257]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    wl = W.Workload("det_varlen", 1, 4, 2, max(lens), D, "bf16", "causal" if causal else "none",
                    varlen=True, n_seqs=len(lens), seed=19)
    T = int(cu[-1])
    g = torch.Generator().manual_seed(19)
    inp = {n: torch.randn(s, generator=g).to(torch.bfloat16) for n, s in
           (("q", (T, 4, D)), ("k", (T, 2, D)), ("v", (T, 2, D)), ("do", (T, 4, D)))}
    inp["cu_seqlens"] = cu
    check_all(wl, gpu_run(wl, inp, deterministic=True), oracle_run(wl, inp, cu=cu))


def test_c3_gqa_sampled_group_deterministic():
    """Causal GQA B=4, 32/8 heads, S=4096 in the deterministic mode: one seeded (b, group) checked."""
    wl = W.WORKLOADS["c3_causal_gqa"]
    inp = W.make_inputs(wl)
    got = gpu_run(wl, inp, deterministic=True)
    rng = np.random.default_rng(77)
    b, g = int(rng.integers(wl.batch)), int(rng.integers(wl.heads_kv))
    G = wl.heads_q // wl.heads_kv
    qh, kh = slice(g * G, (g + 1) * G), slice(g, g + 1)
    ref = oracle_run(wl, _slice_heads(inp, b, qh, kh))
    sub = {"o": got["o"][b:b + 1, qh], "lse": got["lse"][b:b + 1, qh], "dq": got["dq"][b:b + 1, qh],
           "dk": got["dk"][b:b + 1, kh], "dv": got["dv"][b:b + 1, kh]}
    check_all(wl, sub, ref)


def test_c4_block_sparse_sampled_head_deterministic():
    wl = W.WORKLOADS["c4_block_sparse"]
    inp = W.make_inputs(wl)
    got = gpu_run(wl, inp, deterministic=True)
    h = int(np.random.default_rng(88).integers(wl.heads_q))
    ref = oracle_run(wl, _slice_heads(inp, 0, slice(h, h + 1), slice(h, h + 1)))
    check_all(wl, {n: got[n][0:1, h:h + 1] for n in ("o", "lse", "dq", "dk", "dv")}, ref)


def _bwd_twice(wl, inp, deterministic):
    dev = torch.device("cuda")
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    kw = {"scale": wl.scale}
    if wl.mask == "causal":
        kw["causal"] = True
    if wl.mask == "block":
        kw["block_mask"] = BlockMask.from_csr(inp["block_mask"], device=dev)
    if wl.varlen:
        kw["seqlens"] = SeqLens(inp["cu_seqlens"], device=dev)
        kw["seqlen"] = wl.seqlen
    o, lse = attn_fwd(q, k, v, **kw)
    runs = [attn_bwd(q, k, v, o, do, lse, deterministic=deterministic, **kw) for _ in range(2)]
    torch.cuda.synchronize()
    assert get_status() == 0
    return runs


@pytest.mark.parametrize("name", ["h0_causal_s8192", "c5_varlen_causal"])
def test_bit_identical_runs(name):
    """Two deterministic backward calls on a full-size workload give identical bits."""
    wl = W.WORKLOADS[name]
    (dq0, dk0, dv0), (dq1, dk1, dv1) = _bwd_twice(wl, W.make_inputs(wl), deterministic=True)
    for a, b in ((dq0, dq1), (dk0, dk1), (dv0, dv1)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_matches_default_backward_within_tolerance():
    """On the headline dense shape, deterministic and default dQ agree within the bf16 bound."""
    from parity_util import compare
    wl = W.WORKLOADS["h1_dense_s8192"]
    inp = W.make_inputs(wl)
    (dq_d, dk_d, dv_d), _ = _bwd_twice(wl, inp, deterministic=True)
    (dq_a, dk_a, dv_a), _ = _bwd_twice(wl, inp, deterministic=False)
    for n, x, y in (("dq", dq_d, dq_a), ("dk", dk_d, dk_a), ("dv", dv_d, dv_a)):
        compare(f"{n}[det vs default]", x.double().cpu().numpy(), y.double().cpu().numpy(), "bf16")
