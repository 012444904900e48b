"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on the
same seeded inputs, element by element.

Small shapes are compared in full and cover ragged tails, single positions,
GQA, all mask kinds, fully masked rows and variable-length batches with empty
sequences.  The full-size configurations run on the GPU in the benchmark's own
launch configuration and are compared on seeded samples of whole heads (or KV
groups, or sequences) that the oracle computes exactly.
"""

import numpy as np
import pytest
import torch

from bwd_flashattention_fwd_sm_gb300 import workloads as W

from parity_util import check_all, compare, gpu_run, oracle_run

pytestmark = pytest.mark.gpu


def small(name, B, Hq, Hkv, S, D, dtype, mask, seed, **kw):
    return W.Workload(name, B, Hq, Hkv, S, D, dtype, mask, seed=seed, **kw)


def tiles_csr(S, seed, density=0.5, empty_row=None, causal_in_block=1):
    nb = (S + 63) // 64
    rng = np.random.default_rng(seed)
    t = rng.random((nb, nb)) < density
    np.fill_diagonal(t, True)
    if causal_in_block:
        t &= np.tril(np.ones((nb, nb), bool))
    if empty_row is not None and empty_row < nb:
        t[empty_row] = False
    return W.csr_from_dense_blocks(t, causal_in_block=causal_in_block)


SMALL_SHAPES = [(1, 2, 2, 1), (1, 2, 1, 17), (2, 2, 2, 64), (1, 4, 1, 127), (1, 2, 2, 128),
                (2, 4, 4, 129), (1, 8, 2, 300), (1, 16, 1, 257)]


@pytest.mark.parametrize("dtype,D", [("f32", 64), ("f32", 128), ("bf16", 64), ("bf16", 128)])
@pytest.mark.parametrize("mask", ["none", "causal", "block"])
@pytest.mark.parametrize("shape", SMALL_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(shape, mask, dtype, D):
    B, Hq, Hkv, S = shape
    wl = small(f"small_{mask}_{dtype}", B, Hq, Hkv, S, D, dtype, mask, seed=100 + S)
    inp = W.make_inputs(wl.with_(mask="none"))
    if mask == "block":
        inp["block_mask"] = tiles_csr(S, seed=S)
    got = gpu_run(wl, inp)
    ref = oracle_run(wl, inp)
    check_all(wl, got, ref)


@pytest.mark.parametrize("dtype,D", [("f32", 64), ("bf16", 64), ("bf16", 128)])
def test_block_mask_with_empty_row_block(dtype, D):
    """A query block with no listed tile: O = 0, LSE = -inf, no gradient from it."""
    wl = small("empty_row", 1, 2, 2, 256, D, dtype, "block", seed=5)
    inp = W.make_inputs(wl.with_(mask="none"))
    inp["block_mask"] = tiles_csr(256, seed=3, empty_row=2)
    got = gpu_run(wl, inp)
    ref = oracle_run(wl, inp)
    assert np.all(np.isneginf(got["lse"][:, :, 128:192]))
    assert np.all(got["o"][:, :, 128:192] == 0)
    check_all(wl, got, ref)


@pytest.mark.parametrize("dtype,D", [("f32", 64), ("bf16", 64), ("bf16", 128)])
def test_block_mask_without_causal_in_block(dtype, D):
    wl = small("sparse_full", 1, 4, 2, 200, D, dtype, "block", seed=6)
    inp = W.make_inputs(wl.with_(mask="none"))
    inp["block_mask"] = tiles_csr(200, seed=4, density=0.6, causal_in_block=0)
    check_all(wl, gpu_run(wl, inp), oracle_run(wl, inp))


@pytest.mark.parametrize("dtype,D", [("f32", 128), ("bf16", 64), ("bf16", 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_small(causal, dtype, D):
    lens = [5, 0, 128, 1, 200, 64, 129]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    wl = W.Workload("varlen_small", 1, 4, 2, max(lens), D, dtype, "causal" if causal else "none",
                    varlen=True, n_seqs=len(lens), seed=9)
    T = int(cu[-1])
    g = torch.Generator().manual_seed(9)
    dt = W.torch_dtype(wl)
    inp = {n: torch.randn(s, generator=g).to(dt) for n, s in
           (("q", (T, 4, D)), ("k", (T, 2, D)), ("v", (T, 2, D)), ("do", (T, 4, D)))}
    inp["cu_seqlens"] = cu
    got = gpu_run(wl, inp)
    ref = oracle_run(wl, inp, cu=cu)
    check_all(wl, got, ref)


def test_c1_fp32_dense():
    """fp32 config: B=1, H=2, S=64, D=64, no mask; max-abs 1e-3 on every output."""
    wl = W.WORKLOADS["c1_dense_f32"]
    inp = W.make_inputs(wl)
    check_all(wl, gpu_run(wl, inp), oracle_run(wl, inp))


def test_c2_causal_fwd_full():
    """Causal MHA forward, B=2, H=16, S=2048: every head against the oracle."""
    wl = W.WORKLOADS["c2_causal_fwd"]
    inp = W.make_inputs(wl)
    got = gpu_run(wl, inp, passes="fwd")
    ref = oracle_run(wl, inp, passes="fwd")
    check_all(wl, got, ref, names=("o", "lse"))


def _slice_heads(inp, b, qh, kh):
    out = dict(inp)
    for n in ("q", "do"):
        out[n] = inp[n][b:b + 1, qh]
    for n in ("k", "v"):
        out[n] = inp[n][b:b + 1, kh]
    return out


def test_c3_gqa_sampled_group():
    """Causal GQA B=4, 32 q heads / 8 kv heads, S=4096: full run, one seeded (b, kv-group) checked."""
    wl = W.WORKLOADS["c3_causal_gqa"]
    inp = W.make_inputs(wl)
    got = gpu_run(wl, inp)
    rng = np.random.default_rng(33)
    b, g = int(rng.integers(wl.batch)), int(rng.integers(wl.heads_kv))
    G = wl.heads_q // wl.heads_kv
    qh, kh = slice(g * G, (g + 1) * G), slice(g, g + 1)
    ref = oracle_run(wl, _slice_heads(inp, b, qh, kh))
    sub = {"o": got["o"][b:b + 1, qh], "lse": got["lse"][b:b + 1, qh], "dq": got["dq"][b:b + 1, qh],
           "dk": got["dk"][b:b + 1, kh], "dv": got["dv"][b:b + 1, kh]}
    check_all(wl, sub, ref)


def test_c4_block_sparse_sampled_heads():
    """Block-sparse S=8192, H=16: full run, two seeded heads checked."""
    wl = W.WORKLOADS["c4_block_sparse"]
    inp = W.make_inputs(wl)
    got = gpu_run(wl, inp)
    rng = np.random.default_rng(44)
    for h in rng.choice(wl.heads_q, size=2, replace=False):
        h = int(h)
        ref = oracle_run(wl, _slice_heads(inp, 0, slice(h, h + 1), slice(h, h + 1)))
        sub = {n: got[n][0:1, h:h + 1] for n in ("o", "lse", "dq", "dk", "dv")}
        check_all(wl, sub, ref)


def test_c5_varlen_sampled_sequences():
    """Packed 16 sequences, lengths U[128, 8192], H=32, causal: full run, one head of four seeded sequences checked."""
    wl = W.WORKLOADS["c5_varlen_causal"]
    inp = W.make_inputs(wl)
    got = gpu_run(wl, inp)
    cu = inp["cu_seqlens"]
    rng = np.random.default_rng(55)
    h = int(rng.integers(wl.heads_q))
    seqs = sorted(rng.choice(wl.n_seqs, size=4, replace=False).tolist())
    idx = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in seqs])
    lens = [int(cu[n + 1] - cu[n]) for n in seqs]
    sub_cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    sub_in = {n: inp[n][idx][:, h:h + 1] for n in ("q", "k", "v", "do")}
    ref = oracle_run(wl, sub_in, cu=sub_cu)
    sub = {n: got[n][idx][:, h:h + 1] for n in ("o", "dq", "dk", "dv")}
    sub["lse"] = got["lse"][h:h + 1, idx]
    check_all(wl, sub, ref)


@pytest.mark.parametrize("name", ["h0_dense_s8192", "h0_causal_s8192", "h2_dense_s8192_d64", "h2_causal_s8192_d64"])
def test_h0_s8192_sampled_head(name):
    """The S=8192 shapes (B=2, H=16; head dim 128, and 64 with P in tensor-memory
    columns of its own): full run, one seeded head checked."""
    wl = W.WORKLOADS[name]
    inp = W.make_inputs(wl)
    got = gpu_run(wl, inp)
    rng = np.random.default_rng(66)
    b, h = int(rng.integers(wl.batch)), int(rng.integers(wl.heads_q))
    ref = oracle_run(wl, _slice_heads(inp, b, slice(h, h + 1), slice(h, h + 1)))
    sub = {n: got[n][b:b + 1, h:h + 1] for n in ("o", "lse", "dq", "dk", "dv")}
    check_all(wl, sub, ref)


def test_empty_batch():
    from bwd_flashattention_fwd_sm_gb300 import attn_bwd, attn_fwd
    q = torch.zeros((0, 2, 64, 128), dtype=torch.bfloat16, device="cuda")
    o, lse = attn_fwd(q, q, q)
    dq, dk, dv = attn_bwd(q, q, q, o, q, lse)
    assert o.shape == q.shape and lse.shape == (0, 2, 64) and dq.shape == q.shape


def test_longest_sequence_sampled_head():
    """S = 32768 (four times the headline length), causal, D = 64, one head: the
    whole problem on the GPU against the oracle's full result (LSE spans the
    largest row sums, the last query tile sees 256 key tiles)."""
    wl = W.Workload("long_s32768", 1, 1, 1, 32768, 64, "bf16", "causal", seed=13)
    inp = W.make_inputs(wl)
    check_all(wl, gpu_run(wl, inp), oracle_run(wl, inp))
