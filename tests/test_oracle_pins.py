"""Pins for the float64 oracle: checks against facts fixed by the mathematics.

None of these compares the oracle with itself.  Each test states a property that
the plain definition of attention (and the softmax Jacobian for the gradients)
forces, computed here by a different route: hand-derived closed forms, invariants,
a float64 PyTorch library evaluation of the full score matrix with autograd,
central finite differences of L = sum(dO * O), and reductions between mask and
head layouts.  A dropped term, a wrong sign, a transposed operand or a wrong
index in the oracle breaks at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from bwd_flashattention_fwd_sm_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def dense_keep(S, causal=False, tiles=None, block=64, causal_in_block=0):
    """[S, S] boolean keep matrix built by broadcasting (library ops, no loops)."""
    keep = np.ones((S, S), dtype=bool)
    if tiles is not None:
        keep &= np.kron(tiles, np.ones((block, block), dtype=bool)).astype(bool)[:S, :S]
        if causal_in_block:
            keep &= np.tril(np.ones((S, S), dtype=bool))
    if causal:
        keep &= np.tril(np.ones((S, S), dtype=bool))
    return keep


def torch_attention(q, k, v, do, scale, keep):
    """Full-score-matrix attention in float64 with torch autograd.

    q [B, Hq, S, D], k/v [B, Hkv, S, D]; keep [S, S] boolean.  KV heads are
    repeated over their query-head groups; autograd sums the group's gradients.
    """
    G = q.shape[1] // k.shape[1]
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    kk = tk.repeat_interleave(G, dim=1)
    vv = tv.repeat_interleave(G, dim=1)
    s = torch.matmul(tq, kk.transpose(-1, -2)) * scale
    s = s.masked_fill(~torch.tensor(keep), float("-inf"))
    p = torch.softmax(s, dim=-1)
    o = torch.matmul(p, vv)
    lse = torch.logsumexp(s, dim=-1)
    o.backward(torch.tensor(do, dtype=torch.float64))
    return o.detach().numpy(), lse.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


# ---------------------------------------------------------------------------
# Worked example with hand-derived values
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["none", "causal"])
def test_golden_two_keys(mode):
    g = json.load(open(os.path.join(GOLDEN, "two_keys_closed_form.json")))
    inp = g["inputs"]
    sh = (1, 1, 2, 1)
    q, k, v, do = (np.asarray(inp[n], dtype=np.float64).reshape(sh) for n in ("q", "k", "v", "do"))
    causal = mode == "causal"
    o, lse = oracle.attn_fwd(q, k, v, scale=inp["scale"], causal=causal)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, scale=inp["scale"], causal=causal)
    exp = g[mode]
    np.testing.assert_allclose(o.ravel(), np.ravel(exp["o"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse.ravel(), np.ravel(exp["lse"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dq.ravel(), np.ravel(exp["dq"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk.ravel(), np.ravel(exp["dk"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv.ravel(), np.ravel(exp["dv"]), rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# Invariants and closed forms
# ---------------------------------------------------------------------------

MASKS = ["none", "causal", "block"]


def block_tiles_for(S, seed):
    nb = (S + 63) // 64
    rng = np.random.default_rng(seed)
    tiles = rng.random((nb, nb)) < 0.6
    np.fill_diagonal(tiles, True)
    return tiles


@pytest.mark.parametrize("mask", MASKS)
def test_rows_sum_to_one(mask):
    """Softmax rows sum to 1: a V whose column t is the constant c_t gives O[:, t] = c_t."""
    B, Hq, Hkv, S, D = 2, 4, 2, 150, 16
    q, k = rnd((B, Hq, S, D), 1), rnd((B, Hkv, S, D), 2)
    c = np.linspace(-3, 5, D)
    v = np.broadcast_to(c, (B, Hkv, S, D)).copy()
    kw = {}
    if mask == "causal":
        kw["causal"] = True
    if mask == "block":
        kw["block_mask"] = W.csr_from_dense_blocks(block_tiles_for(S, 3), causal_in_block=1)
    o, lse = oracle.attn_fwd(q, k, v, scale=0.3, **kw)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-12)
    assert np.all(np.isfinite(lse))


@pytest.mark.parametrize("mask", ["none", "causal", "diag_block", "lower_blocks"])
def test_identical_keys_give_mean_of_v(mask):
    """All keys equal: every allowed score is s, so O_i = mean of allowed v_j, LSE_i = s + ln|A_i|."""
    B, H, S, D = 1, 2, 200, 8
    q = rnd((B, H, S, D), 4)
    k = np.broadcast_to(rnd((1, 1, 1, D), 5), (B, H, S, D)).copy()
    v = rnd((B, H, S, D), 6)
    scale = 0.7
    nb = (S + 63) // 64
    i = np.arange(S)
    kw = {}
    if mask == "none":
        count = np.full(S, S)
        first = np.zeros(S, dtype=int)
    elif mask == "causal":
        kw["causal"] = True
        count = i + 1
        first = np.zeros(S, dtype=int)
    elif mask == "diag_block":  # only the diagonal tile, causal inside it
        kw["block_mask"] = W.csr_from_dense_blocks(np.eye(nb, dtype=bool), causal_in_block=1)
        count = i % 64 + 1
        first = (i // 64) * 64
    else:  # every tile on or below the diagonal, causal inside: same as causal
        kw["block_mask"] = W.csr_from_dense_blocks(np.tril(np.ones((nb, nb), bool)), causal_in_block=1)
        count = i + 1
        first = np.zeros(S, dtype=int)
    o, lse = oracle.attn_fwd(q, k, v, scale=scale, **kw)
    csum = np.cumsum(v, axis=2)
    for b in range(B):
        for h in range(H):
            last = first + count - 1
            tot = csum[b, h, last] - np.where(first[:, None] > 0, csum[b, h, np.maximum(first - 1, 0)], 0.0)
            np.testing.assert_allclose(o[b, h], tot / count[:, None], rtol=0, atol=1e-12)
            s = scale * q[b, h] @ k[b, h, 0]
            np.testing.assert_allclose(lse[b, h], s + np.log(count), rtol=0, atol=1e-12)


def test_single_allowed_key_is_exact():
    """A row with one allowed key returns that key's V row exactly, LSE = its score, dQ = 0."""
    B, H, S, D = 1, 2, 130, 8
    q, k, v, do = rnd((B, H, S, D), 7), rnd((B, H, S, D), 8), rnd((B, H, S, D), 9), rnd((B, H, S, D), 10)
    scale = 0.4
    nb = (S + 63) // 64
    bm = W.csr_from_dense_blocks(np.eye(nb, dtype=bool), causal_in_block=1)
    for kw, rows in (({"causal": True}, [0]), ({"block_mask": bm}, [0, 64, 128])):
        o, lse = oracle.attn_fwd(q, k, v, scale=scale, **kw)
        dq, _, _ = oracle.attn_bwd(q, k, v, do, scale=scale, **kw)
        for r in rows:
            assert np.array_equal(o[:, :, r], v[:, :, r])
            np.testing.assert_allclose(lse[:, :, r], scale * np.einsum("bhd,bhd->bh", q[:, :, r], k[:, :, r]),
                                       rtol=0, atol=1e-14)
            assert np.all(dq[:, :, r] == 0.0)


def test_scale_zero_gives_mean_of_allowed_v():
    B, H, S, D = 1, 3, 77, 16
    q, k, v = rnd((B, H, S, D), 11), rnd((B, H, S, D), 12), rnd((B, H, S, D), 13)
    o, lse = oracle.attn_fwd(q, k, v, scale=0.0, causal=True)
    cm = np.cumsum(v, axis=2) / np.arange(1, S + 1)[None, None, :, None]
    np.testing.assert_allclose(o, cm, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, S + 1)), lse.shape), rtol=0, atol=1e-12)
    o, _ = oracle.attn_fwd(q, k, v, scale=0.0)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), rtol=0, atol=1e-12)


def test_fully_masked_row():
    """A row block with no listed tile: O = 0, LSE = -inf, and no gradient flows through it."""
    B, H, S, D = 1, 2, 128, 8
    q, k, v, do = rnd((B, H, S, D), 14), rnd((B, H, S, D), 15), rnd((B, H, S, D), 16), rnd((B, H, S, D), 17)
    tiles = np.array([[True, False], [False, False]])
    bm = W.csr_from_dense_blocks(tiles)
    o, lse = oracle.attn_fwd(q, k, v, scale=0.3, block_mask=bm)
    assert np.all(o[:, :, 64:] == 0) and np.all(np.isneginf(lse[:, :, 64:]))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, scale=0.3, block_mask=bm)
    assert np.all(dq[:, :, 64:] == 0) and np.all(dk[:, :, 64:] == 0) and np.all(dv[:, :, 64:] == 0)
    # the first row block alone is plain dense attention over the first 64 keys
    o2, _ = oracle.attn_fwd(q[:, :, :64], k[:, :, :64], v[:, :, :64], scale=0.3)
    np.testing.assert_allclose(o[:, :, :64], o2, rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# Streamed online softmax reaches the plain definition
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("block", [1, 7, 64])
@pytest.mark.parametrize("mask", MASKS)
def test_blocked_equals_unblocked(block, mask):
    B, Hq, Hkv, S, D = 1, 4, 2, 140, 16
    q, k, v = rnd((B, Hq, S, D), 20), rnd((B, Hkv, S, D), 21), rnd((B, Hkv, S, D), 22)
    q *= 3.0  # wide score range so the running-max correction matters
    kw = {}
    if mask == "causal":
        kw["causal"] = True
    if mask == "block":
        kw["block_mask"] = W.csr_from_dense_blocks(block_tiles_for(S, 23), causal_in_block=1)
    o1, l1 = oracle.attn_fwd(q, k, v, scale=0.25, **kw)
    o2, l2 = oracle.attn_fwd_blocked(q, k, v, scale=0.25, block=block, **kw)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Library cross-check: full score matrix in torch float64 with autograd
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("shape", [(1, 2, 2, 64, 64), (2, 4, 1, 129, 32), (1, 6, 3, 17, 8)])
def test_matches_torch_float64(mask, shape):
    B, Hq, Hkv, S, D = shape
    q, k, v, do = rnd((B, Hq, S, D), 30), rnd((B, Hkv, S, D), 31), rnd((B, Hkv, S, D), 32), rnd((B, Hq, S, D), 33)
    scale = 1.0 / math.sqrt(D)
    kw = {}
    if mask == "none":
        keep = dense_keep(S)
    elif mask == "causal":
        kw["causal"] = True
        keep = dense_keep(S, causal=True)
    else:
        tiles = block_tiles_for(S, 34)
        kw["block_mask"] = W.csr_from_dense_blocks(tiles, causal_in_block=1)
        keep = dense_keep(S, tiles=tiles, causal_in_block=1)
    o, lse = oracle.attn_fwd(q, k, v, scale=scale, **kw)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, scale=scale, **kw)
    to, tl, tdq, tdk, tdv = torch_attention(q, k, v, do, scale, keep)
    for a, b in ((o, to), (lse, tl), (dq, tdq), (dk, tdk), (dv, tdv)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)


def test_c1_config_matches_torch_float64():
    """The fp32 configuration's shape (B=1, H=2, S=64, D=64, no mask) on its own seeded inputs."""
    wl = W.WORKLOADS["c1_dense_f32"]
    t = W.make_inputs(wl)
    q, k, v, do = (t[n].double().numpy() for n in ("q", "k", "v", "do"))
    o, lse = oracle.attn_fwd(q, k, v, scale=wl.scale)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, scale=wl.scale)
    to, tl, tdq, tdk, tdv = torch_attention(q, k, v, do, wl.scale, dense_keep(wl.seqlen))
    for a, b in ((o, to), (lse, tl), (dq, tdq), (dk, tdk), (dv, tdv)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)


# ---------------------------------------------------------------------------
# Finite differences of L = sum(dO * O)
# ---------------------------------------------------------------------------

def _fd_check(q, k, v, do, scale, cu=None, **kw):
    h = 1e-6

    def loss(q_, k_, v_):
        o, _ = oracle.attn_fwd(q_, k_, v_, scale=scale, cu_seqlens=cu, nthreads=1, **kw)
        return float(np.sum(do * o))

    dq, dk, dv = oracle.attn_bwd(q, k, v, do, scale=scale, cu_seqlens=cu, nthreads=1, **kw)
    for which, (arr, grad) in enumerate(((q, dq), (k, dk), (v, dv))):
        num = np.zeros_like(arr)
        flat = arr.reshape(-1)
        for idx in range(flat.size):
            old = flat[idx]
            flat[idx] = old + h
            lp = loss(q, k, v)
            flat[idx] = old - h
            lm = loss(q, k, v)
            flat[idx] = old
            num.reshape(-1)[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(num - grad)) / max(1.0, np.max(np.abs(grad)))
        assert err <= 1e-6, f"gradient {'qkv'[which]}: relative error {err:.3e}"


@pytest.mark.parametrize("G", [1, 2])
@pytest.mark.parametrize("mask", MASKS)
def test_finite_differences_fixed(G, mask):
    B, Hq, S, D = 1, 2, 9, 8
    Hkv = Hq // G
    q, k, v, do = rnd((B, Hq, S, D), 40), rnd((B, Hkv, S, D), 41), rnd((B, Hkv, S, D), 42), rnd((B, Hq, S, D), 43)
    kw = {}
    if mask == "causal":
        kw["causal"] = True
    if mask == "block":
        # 4-token tiles so that S=9 spans a 3x3 tile map with holes
        tiles = np.array([[1, 0, 0], [1, 1, 0], [0, 1, 1]], dtype=bool)
        bm = W.csr_from_dense_blocks(tiles, block=4, causal_in_block=1)
        kw["block_mask"] = bm
    _fd_check(q, k, v, do, 0.35, **kw)


@pytest.mark.parametrize("G", [1, 2])
def test_finite_differences_varlen(G):
    lens = [3, 1, 5]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, Hq, D = int(cu[-1]), 2, 6
    Hkv = Hq // G
    q, k, v, do = rnd((T, Hq, D), 44), rnd((T, Hkv, D), 45), rnd((T, Hkv, D), 46), rnd((T, Hq, D), 47)
    _fd_check(q, k, v, do, 0.5, cu=cu, causal=True)


# ---------------------------------------------------------------------------
# Reductions between layouts
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_mha_with_repeated_kv(causal):
    B, Hq, Hkv, S, D = 2, 8, 2, 70, 16
    G = Hq // Hkv
    q, k, v, do = rnd((B, Hq, S, D), 50), rnd((B, Hkv, S, D), 51), rnd((B, Hkv, S, D), 52), rnd((B, Hq, S, D), 53)
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    o1, l1 = oracle.attn_fwd(q, k, v, scale=0.2, causal=causal)
    o2, l2 = oracle.attn_fwd(q, kr, vr, scale=0.2, causal=causal)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)
    g1 = oracle.attn_bwd(q, k, v, do, scale=0.2, causal=causal)
    g2 = oracle.attn_bwd(q, kr, vr, do, scale=0.2, causal=causal)
    np.testing.assert_allclose(g1[0], g2[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(g1[1], g2[1].reshape(B, Hkv, G, S, D).sum(axis=2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(g1[2], g2[2].reshape(B, Hkv, G, S, D).sum(axis=2), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_each_sequence_alone(causal):
    lens = [5, 64, 1, 130, 33]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, Hq, Hkv, D = int(cu[-1]), 4, 2, 16
    q, k, v, do = rnd((T, Hq, D), 60), rnd((T, Hkv, D), 61), rnd((T, Hkv, D), 62), rnd((T, Hq, D), 63)
    o, lse = oracle.attn_fwd(q, k, v, scale=0.25, causal=causal, cu_seqlens=cu)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, scale=0.25, causal=causal, cu_seqlens=cu)
    for n, L in enumerate(lens):
        sl = slice(cu[n], cu[n + 1])
        tr = lambda a: a[sl].transpose(1, 0, 2)[None]  # [L, H, D] -> [1, H, L, D]
        o1, l1 = oracle.attn_fwd(tr(q), tr(k), tr(v), scale=0.25, causal=causal)
        g1 = oracle.attn_bwd(tr(q), tr(k), tr(v), tr(do), scale=0.25, causal=causal)
        np.testing.assert_allclose(tr(o), o1, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, sl][None], l1, rtol=0, atol=1e-13)
        for a, b in zip((dq, dk, dv), g1):
            np.testing.assert_allclose(tr(a), b, rtol=0, atol=1e-12)


def test_block_mask_reductions():
    B, H, S, D = 1, 2, 192, 16
    q, k, v, do = rnd((B, H, S, D), 70), rnd((B, H, S, D), 71), rnd((B, H, S, D), 72), rnd((B, H, S, D), 73)
    nb = S // 64
    lower = W.csr_from_dense_blocks(np.tril(np.ones((nb, nb), bool)), causal_in_block=1)
    full = W.csr_from_dense_blocks(np.ones((nb, nb), bool), causal_in_block=0)
    for bm, causal in ((lower, True), (full, False)):
        o1, l1 = oracle.attn_fwd(q, k, v, scale=0.3, block_mask=bm)
        o2, l2 = oracle.attn_fwd(q, k, v, scale=0.3, causal=causal)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
        np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)
        g1 = oracle.attn_bwd(q, k, v, do, scale=0.3, block_mask=bm)
        g2 = oracle.attn_bwd(q, k, v, do, scale=0.3, causal=causal)
        for a, b in zip(g1, g2):
            np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Workload generators (input side only)
# ---------------------------------------------------------------------------

def test_c4_mask_structure():
    wl = W.WORKLOADS["c4_block_sparse"]
    bm = W.block_mask_csr(wl)
    nb = bm["n_row_blocks"]
    assert nb == 128
    rp, ci = bm["row_ptr"], bm["col_idx"]
    for i in range(nb):
        cols = ci[rp[i]:rp[i + 1]]
        assert np.all(np.diff(cols) > 0) and cols.max() <= i
        assert set(range(max(0, i - 15), i + 1)) <= set(cols.tolist())
    nnz = int(rp[-1])
    assert 4500 < nnz < 5700, nnz  # about 31% of the 16384 tiles


def test_unmasked_pairs_counts():
    wl = W.WORKLOADS["h0_causal_s8192"]
    assert W.unmasked_pairs(wl) == 2 * 8192 * 8193 // 2
    wl = W.Workload("t", 1, 1, 1, 256, 64, "bf16", "block", seed=9)
    bm = W.csr_from_dense_blocks(np.tril(np.ones((4, 4), bool)), causal_in_block=1)
    assert W.unmasked_pairs(wl, bm) == 256 * 257 // 2
