"""GPU parity of the FP8 (e4m3) forward against the oracle (oracle/fp8.py).

attn_quantize_fp8: codes and scales bit-identical to the oracle's per-tile
quantisation (each code is decided in float32 on both sides).

attn_fwd_fp8, against the float64 attention on the dequantised inputs (the
oracle quantises the bf16 inputs itself; nothing on its side comes from the GPU):
  LSE within 1e-3: it comes from the unrounded P, so only float32 rounding
      separates it from the oracle's;
  O per element within the P-rounding bound (oracle/fp8.p_rounding_bound) plus
      the bf16 rounding of O (at most 2^-8 of the value: half a unit in the
      last of 8 significant bits) and float32 slack of 2^-12 of
      A = sum_j P_ij |v_jd| (float32 sums over n keys are off by at most
      n 2^-24 A; 2^-12 covers n up to 4096 and the sampled 8192-key rows in
      practice);
  O relative L2 error at most 2^-4: rounding moves every normal-range P by at
      most 2^-4 of itself (the float64 replay of the kernel's order gives 0.037).
Inputs: N(0, 1) with each 128-row tile scaled by 2^U{-3..3}, so that a scale
taken from the wrong tile would change results by up to 64x.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as ofp8
from bwd_flashattention_fwd_sm_gb300 import BlockMask, attn_fwd_fp8, get_status, make_params, quantize_fp8
from bwd_flashattention_fwd_sm_gb300 import _lib
from bwd_flashattention_fwd_sm_gb300 import workloads as W
from bwd_flashattention_fwd_sm_gb300.attention import Fp8Operands

from parity_util import _log_margin

from test_gpu_parity import tiles_csr

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]

DEV = torch.device("cuda", 0)


def _inputs(B, Hq, Hkv, S, seed, spread=3):
    inp = W.make_inputs(W.Workload("fp8", B, Hq, Hkv, S, 128, "bf16", "none", seed=seed))
    return tuple(W.tile_spread(inp[n], seed + i, spread) for i, n in enumerate(("q", "k", "v"), 1))


def _oracle_quant(x):
    codes, scales = ofp8.quantize_tiles(x.float().numpy())
    return codes, scales, ofp8.dequantize(codes, scales)


def _check_fwd(o, lse, q, k, v, *, scale, causal=False, csr=None):
    _, _, qd = _oracle_quant(q)
    _, _, kd = _oracle_quant(k)
    _, vs, vd = _oracle_quant(v)
    ro, rl = oracle.attn_fwd(qd, kd, vd, scale=scale, causal=causal, block_mask=csr)
    terms, A = ofp8.p_rounding_bound(qd, kd, vd, vs, scale=scale, causal=causal, block_mask=csr)
    _compare(o, lse, ro, rl, terms, A)


def _compare(o, lse, ro, rl, terms, A, name="fp8"):
    go = o.double().cpu().numpy()
    gl = lse.double().cpu().numpy()
    assert np.array_equal(np.isneginf(gl), np.isneginf(rl))
    fin = np.isfinite(rl)
    lse_err = float(np.abs(gl[fin] - rl[fin]).max()) if np.any(fin) else 0.0
    tol = terms * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(ro) + 2.0 ** -12 * A + 1e-6
    err = np.abs(go - ro)
    nr = np.linalg.norm(ro)
    rel = float(np.linalg.norm(go - ro) / nr) if nr > 0 else 0.0
    _log_margin(f"o[{name}]", "fp8", float(err.max()), rel, float(np.max(err / tol)), err.size)
    _log_margin(f"lse[{name}]", "fp8", lse_err, 0.0, lse_err / 1e-3, int(np.sum(fin)))
    assert lse_err <= 1e-3, lse_err
    assert np.all(err <= tol), f"max err/tol {np.max(err / tol):.3f}"
    if nr > 0:
        assert rel <= 2.0 ** -4


QUANT_SHAPES = [(1, 2, 1, 1), (1, 1, 1, 16), (1, 1, 1, 17), (1, 2, 2, 100), (1, 2, 1, 129), (2, 4, 2, 300),
                (1, 3, 1, 1000)]


@pytest.mark.parametrize("shape", QUANT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_quantize_bit_exact(shape):
    B, Hq, Hkv, S = shape
    q, k, v = _inputs(B, Hq, Hkv, S, seed=300 + S)
    f = quantize_fp8(q.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    assert get_status() == 0
    for name, x, codes, scales in (("q", q, f.q8, f.q_scale), ("k", k, f.k8, f.k_scale)):
        rc, rs, _ = _oracle_quant(x)
        assert np.array_equal(codes.cpu().numpy(), rc), name
        assert np.array_equal(scales.cpu().numpy(), rs), name
    rc, rs, _ = _oracle_quant(v)
    vt = f.v8t.cpu().numpy()[..., :S]  # [B, Hkv, 128, S]: keys along rows
    assert np.array_equal(vt.transpose(0, 1, 3, 2), rc)
    assert np.array_equal(f.v_scale.cpu().numpy(), rs)


def test_quantize_zero_tile_and_strided_input():
    """Position-major (BSHD) inputs through the strides; an all-zero tile gets scale 0."""
    B, H, S = 1, 2, 260
    q, k, v = _inputs(B, H, H, S, seed=41)
    q[:, 1, 128:256] = 0
    qs, ks, vs_ = (t.transpose(1, 2).contiguous().to(DEV) for t in (q, k, v))  # [B, S, H, D]
    qv, kv, vv = (t.transpose(1, 2) for t in (qs, ks, vs_))                     # [B, H, S, D] views
    p = make_params(qv, kv)
    f = Fp8Operands.empty(B, H, H, S, DEV)
    lib = _lib.load()
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.attn_quantize_fp8(ctypes.byref(p), ptr(qv), ptr(kv), ptr(vv), ptr(f.q8), ptr(f.k8), ptr(f.v8t),
                               ptr(f.q_scale), ptr(f.k_scale), ptr(f.v_scale),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _lib.ATTN_OK
    torch.cuda.synchronize()
    rc_q, rs_q, _ = _oracle_quant(q)
    assert rs_q[0, 1, 1] == 0 and f.q_scale[0, 1, 1].item() == 0
    assert np.array_equal(f.q8.cpu().numpy(), rc_q) and np.array_equal(f.q_scale.cpu().numpy(), rs_q)
    rc_v, rs_v, _ = _oracle_quant(v)
    assert np.array_equal(f.v8t.cpu().numpy()[..., :S].transpose(0, 1, 3, 2), rc_v)


FWD_CASES = [(1, 2, 1, 1, "none"), (1, 2, 2, 100, "causal"), (2, 4, 2, 300, "none"), (1, 4, 1, 513, "causal"),
             (1, 2, 2, 640, "block"), (1, 2, 1, 1000, "none"), (2, 2, 2, 129, "block"), (1, 16, 1, 257, "causal")]


@pytest.mark.parametrize("case", FWD_CASES, ids=lambda c: "x".join(map(str, c)))
def test_fwd_fp8_parity(case):
    B, Hq, Hkv, S, mask = case
    q, k, v = _inputs(B, Hq, Hkv, S, seed=400 + S + Hq)
    csr = tiles_csr(S, seed=S + 3) if mask == "block" else None
    scale = 1.0 / np.sqrt(128)
    f = quantize_fp8(q.to(DEV), k.to(DEV), v.to(DEV))
    bm = BlockMask.from_csr(csr, device=DEV) if csr is not None else None
    o, lse = attn_fwd_fp8(f, causal=mask == "causal", block_mask=bm, scale=scale)
    o2, lse2 = attn_fwd_fp8(f, causal=mask == "causal", block_mask=bm, scale=scale)
    torch.cuda.synchronize()
    assert get_status() == 0
    assert torch.equal(o, o2) and torch.equal(lse, lse2)  # no atomics: identical from run to run
    _check_fwd(o, lse, q, k, v, scale=scale, causal=mask == "causal", csr=csr)


def test_fwd_fp8_block_mask_empty_row():
    """A query block with no listed tile: O = 0 and LSE = -inf on its rows."""
    S = 384
    q, k, v = _inputs(1, 2, 1, S, seed=77)
    csr = tiles_csr(S, seed=9, empty_row=2)
    f = quantize_fp8(q.to(DEV), k.to(DEV), v.to(DEV))
    o, lse = attn_fwd_fp8(f, block_mask=BlockMask.from_csr(csr, device=DEV), scale=0.1)
    torch.cuda.synchronize()
    assert torch.all(o[:, :, 128:192] == 0) and torch.all(torch.isneginf(lse[:, :, 128:192]))
    _check_fwd(o, lse, q, k, v, scale=0.1, csr=csr)


def test_fwd_fp8_empty_batch():
    f = Fp8Operands.empty(0, 2, 1, 64, DEV)
    o, lse = attn_fwd_fp8(f, causal=True)
    assert o.shape == (0, 2, 64, 128) and lse.shape == (0, 2, 64)


@pytest.mark.parametrize("mask,b,h", [("none", 1, 5), ("causal", 0, 12)])
def test_fwd_fp8_full_size_sampled_rows(mask, b, h):
    """B = 2, H = 16, S = 8192, D = 128: the whole problem on the GPU, one head's
    sampled rows against the oracle (one full head of the float64 reference)."""
    wl = W.Workload("h0_fp8", 2, 16, 16, 8192, 128, "bf16", mask, seed=6)
    inp = W.make_inputs(wl)
    q, k, v = inp["q"], inp["k"], inp["v"]
    f = quantize_fp8(q.to(DEV), k.to(DEV), v.to(DEV))
    o, lse = attn_fwd_fp8(f, causal=mask == "causal", scale=wl.scale)
    torch.cuda.synchronize()
    assert get_status() == 0
    sl = slice(b, b + 1), slice(h, h + 1)
    _, _, qd = _oracle_quant(q[sl])
    _, _, kd = _oracle_quant(k[sl])
    _, vs, vd = _oracle_quant(v[sl])
    ro, rl = oracle.attn_fwd(qd, kd, vd, scale=wl.scale, causal=mask == "causal")
    rows = np.sort(np.random.default_rng(h).choice(8192, 384, replace=False))
    rows[:2] = [0, 1]
    rows[-1] = 8191
    terms, A = ofp8.p_rounding_bound(qd[:, :, rows], kd, vd, vs, scale=wl.scale, causal=mask == "causal",
                                     q_pos=rows)
    _compare(o[sl][:, :, rows], lse[sl][:, :, rows], ro[:, :, rows], rl[:, :, rows], terms, A,
             name=f"h0_fp8 {mask} full size")


@pytest.mark.parametrize("S,causal", [(300, False), (300, True), (1000, True)])
def test_fwd_fp8_exact_when_rounding_is_exact(S, causal):
    """All keys equal, so every allowed P in a row is equal, and V tiles whose
    largest magnitudes differ by powers of two, so every V scale ratio r_j is a
    power of two >= 2^-6: P r_j is then exact in e4m3, and O must equal the mean
    of the allowed dequantised V rows up to the bf16 rounding of O (2^-8 of the
    value) and float32 sums (at most n 2^-24 of sum_j P_ij |v_jd| over n keys).
    This pins the V layout, the per-tile V scales and the P layout in
    tensor memory exactly, where the general bound leaves room."""
    B, Hq, Hkv = 1, 2, 1
    q, k, v = _inputs(B, Hq, Hkv, S, seed=500 + S)
    k[:] = k[:, :, :1, :]
    v = v.float().clamp(-3.5, 3.5)
    v[:, :, ::128, 0] = 4.0  # every tile's amax is 4 before the spread
    v = W.tile_spread(v.to(torch.bfloat16), seed=501, spread=3)
    f = quantize_fp8(q.to(DEV), k.to(DEV), v.to(DEV))
    o, lse = attn_fwd_fp8(f, causal=causal, scale=0.125)
    torch.cuda.synchronize()
    _, _, qd = _oracle_quant(q)
    _, _, kd = _oracle_quant(k)
    _, vs, vd = _oracle_quant(v)
    ratios = vs[0, 0] / vs[0, 0].max()
    assert np.all(np.exp2(np.round(np.log2(ratios))) == ratios) and ratios.min() >= 2.0 ** -6
    ro, rl = oracle.attn_fwd(qd, kd, vd, scale=0.125, causal=causal)
    go = o.double().cpu().numpy()
    allowed = np.tril(np.ones((S, S))) if causal else np.ones((S, S))
    A = np.einsum("ij,bhjd->bhid", allowed / allowed.sum(1, keepdims=True), np.abs(vd)[:, [0, 0]])
    tol = 2.0 ** -8 * np.abs(ro) + S * 2.0 ** -24 * A + 1e-7
    assert np.all(np.abs(go - ro) <= tol), np.max(np.abs(go - ro) / tol)
    assert np.all(np.abs(lse.double().cpu().numpy() - rl) <= 1e-4)
