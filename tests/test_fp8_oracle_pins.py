"""Pins for the FP8 oracle (oracle/fp8.py), on the CPU.

The pages fix no FP8 format or example values, so the oracle is pinned to
things outside itself: the format's closed forms (largest finite value,
smallest subnormal, the NaN codes), PyTorch's own float32 -> float8_e4m3fn
conversion (round to nearest even) over every representable value, every
midpoint and random values, invariants of per-tile scaling that a wrong tile
index or a global scale would break, and the P-rounding bound checked against
a float64 simulation of the blocked, lazily rescaled kernel order.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_decode_closed_forms():
    codes = np.arange(256, dtype=np.uint8)
    vals = fp8.e4m3_decode(codes)
    assert vals[0x7E] == 448.0
    assert vals[0x01] == 2.0 ** -9
    assert vals[0x07] == 7 * 2.0 ** -9
    assert vals[0x08] == 2.0 ** -6
    assert vals[0x38] == 1.0
    assert vals[0x39] == 1.125
    assert vals[0xFE] == -448.0
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    assert np.signbit(vals[0x80]) and vals[0x80] == 0.0
    assert np.count_nonzero(np.isfinite(vals)) == 254
    pos = vals[:0x7F]
    assert np.all(np.diff(pos) > 0)  # codes 0..126 increase strictly


def test_encode_decode_round_trip():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = fp8.e4m3_decode(codes)
    assert np.array_equal(fp8.e4m3_encode(vals), codes)
    assert np.array_equal(fp8.e4m3_round(vals.astype(np.float32)), vals)


def _torch_e4m3(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_round_matches_torch_on_values_midpoints_and_random():
    vals = fp8.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[1:] + vals[:-1]) / 2  # exact in float32: ties, rounded to even
    rng = np.random.default_rng(31)
    mag = np.exp2(rng.uniform(-14, np.log2(464.0), 20000))
    rand = mag * rng.choice([-1.0, 1.0], mag.size)
    for x in (vals, -vals, mids, -mids, rand):
        x32 = np.asarray(x, dtype=np.float32)
        assert np.array_equal(fp8.e4m3_round(x32), _torch_e4m3(x32))


def test_round_saturates():
    x = np.array([464.0, 464.1, 479.0, 500.0, 1e30, np.inf, -500.0, -np.inf], dtype=np.float32)
    out = fp8.e4m3_round(x)
    assert np.array_equal(out, [448, 448, 448, 448, 448, 448, -448, -448])


def test_ties_go_to_even():
    # 1 + 1/16 lies halfway between 1 (mantissa 000) and 1.125 (001): even is 1
    # 1.1875 lies halfway between 1.125 (001) and 1.25 (010): even is 1.25
    out = fp8.e4m3_round(np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10], dtype=np.float32))
    assert np.array_equal(out, [1.0, 1.25, 0.0, 2.0 ** -8])


def _tiles_input(seed, shape, spread=3):
    """Random N(0, 1) bf16 values with each 128-row tile scaled by 2^U{-spread..spread}."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=g)
    nt = (shape[-2] + 127) // 128
    f = torch.pow(2.0, torch.randint(-spread, spread + 1, shape[:-2] + (nt,), generator=g).float())
    x = x * f.repeat_interleave(128, dim=-1)[..., : shape[-2], None]
    return x.to(torch.bfloat16).float().numpy()


def test_quantize_tile_max_is_448_and_error_bounded():
    x = _tiles_input(1, (2, 3, 300, 128))
    codes, scales = fp8.quantize_tiles(x)
    assert codes.shape == x.shape and scales.shape == (2, 3, 3)
    vals = fp8.e4m3_decode(codes)
    for t in range(3):
        blk = np.abs(vals[:, :, t * 128:(t + 1) * 128])
        assert np.all(blk.max(axis=(2, 3)) == 448.0)
    deq = fp8.dequantize(codes, scales)
    sc = np.repeat(scales.astype(np.float64), 128, axis=-1)[..., :300, None]
    # float32 scaling (relative 2^-23) then e4m3 rounding (relative 2^-4 above
    # 2^-6, absolute 2^-10 in code units below)
    bound = (2.0 ** -4 + 2.0 ** -20) * np.abs(x) + 2.0 ** -10 * sc
    assert np.all(np.abs(deq - x) <= bound)


def test_quantize_scale_is_per_tile():
    x = _tiles_input(2, (1, 2, 384, 128))
    codes, scales = fp8.quantize_tiles(x)
    # another tile's values do not change this tile
    y = x.copy()
    y[:, :, 128:256] *= 3.0
    c2, s2 = fp8.quantize_tiles(y)
    assert np.array_equal(c2[:, :, :128], codes[:, :, :128]) and np.array_equal(c2[:, :, 256:], codes[:, :, 256:])
    assert np.array_equal(s2[..., [0, 2]], scales[..., [0, 2]])
    # a power-of-two factor on one tile moves only its scale
    z = x.copy()
    z[:, :, 256:] *= 8.0
    c3, s3 = fp8.quantize_tiles(z)
    assert np.array_equal(c3, codes)
    assert np.array_equal(s3[..., 2], scales[..., 2] * 8) and np.array_equal(s3[..., :2], scales[..., :2])
    # row order inside a tile does not change its scale; rows move with their codes
    perm = np.random.default_rng(3).permutation(128)
    w = x.copy()
    w[:, :, :128] = x[:, :, perm]
    c4, s4 = fp8.quantize_tiles(w)
    assert np.array_equal(s4, scales) and np.array_equal(c4[:, :, :128], codes[:, :, perm])


def test_quantize_zero_and_ragged_tiles():
    x = np.zeros((1, 1, 130, 128), dtype=np.float32)
    x[0, 0, 129, 5] = -2.0
    codes, scales = fp8.quantize_tiles(x)
    assert scales[0, 0, 0] == 0.0 and not codes[0, 0, :128].any()
    assert scales[0, 0, 1] == np.float32(2.0) / np.float32(448.0)
    assert fp8.e4m3_decode(codes[0, 0, 129, 5]) == -448.0
    assert np.count_nonzero(codes) == 1


def _simulate_kernel(qd, kd, vcodes, vscales, scale, causal):
    """float64 replay of the GPU's blocked forward with P rounded to e4m3.

    Key tiles of 128 in ascending order; running max in log2 units, the output
    rescaled only when the maximum grows by more than 8; p = 2^(x - m_used) r_j
    rounded to e4m3 for the P V product; the row sum from the unrounded p / r_j.
    """
    B, Hq, S, D = qd.shape
    G = Hq // kd.shape[1]
    out = np.zeros_like(qd)
    c = scale / np.log(2.0)
    cv = fp8.e4m3_decode(vcodes)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            ref = vscales[b, g].max()
            x_all = c * (qd[b, h] @ kd[b, g].T)
            for i in range(S):
                m_used, l, acc = -np.inf, 0.0, np.zeros(D)
                for t in range((S + 127) // 128):
                    lo, hi = t * 128, min(S, t * 128 + 128)
                    x = x_all[i, lo:hi].copy()
                    keep = np.arange(lo, hi) <= i if causal else np.ones(hi - lo, bool)
                    if not keep.any():
                        continue
                    mx = x[keep].max()
                    if mx > m_used + 8:
                        if np.isfinite(m_used):
                            alpha = 2.0 ** (m_used - mx)
                            l *= alpha
                            acc *= alpha
                        m_used = mx
                    r = vscales[b, g, t] / ref if ref > 0 else 1.0
                    p = np.where(keep, 2.0 ** (x - m_used), 0.0)
                    pq = fp8.e4m3_round((p * r).astype(np.float32))
                    acc += pq @ cv[b, g, lo:hi]
                    l += p.sum()
                out[b, h, i] = acc * ref / l if l > 0 else 0.0
    return out


@pytest.mark.parametrize("causal,sc", [(False, None), (True, None), (False, 0.6)])
def test_p_rounding_bound_holds_on_simulated_kernel(causal, sc):
    q = _tiles_input(5, (1, 2, 260, 128), spread=1)
    k = _tiles_input(6, (1, 1, 260, 128), spread=1)
    v = _tiles_input(7, (1, 1, 260, 128), spread=3)
    scale = sc if sc is not None else 1 / np.sqrt(128)  # 0.6: peaky rows, most P below 2^-10
    q8, qs = fp8.quantize_tiles(q)
    k8, ks = fp8.quantize_tiles(k)
    v8, vs = fp8.quantize_tiles(v)
    qd, kd, vd = fp8.dequantize(q8, qs), fp8.dequantize(k8, ks), fp8.dequantize(v8, vs)
    ref, _ = oracle.attn_fwd(qd, kd, vd, scale=scale, causal=causal)
    sim = _simulate_kernel(qd, kd, v8, vs, scale, causal)
    terms, A = fp8.p_rounding_bound(qd, kd, vd, vs, scale=scale, causal=causal)
    err = np.abs(sim - ref)
    assert np.all(err <= terms * (1 + 1e-9) + 1e-12)
    assert err.max() > 0  # the rounding does act
    # the typical error is far inside the worst case: random rounding errors cancel
    rel = np.linalg.norm(sim - ref) / np.linalg.norm(ref)
    assert rel < 0.05
