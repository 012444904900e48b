"""Oracle for the FP8 (e4m3) attention forward: quantisation and reference.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``): only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may use it.

Why FP8.  The smzdm contest article ("杀进决赛!这 28 支队伍把算子优化卷疯了!",
closing section on precision) says newer accelerators compute with 8-bit floats,
so each transfer and each matrix instruction handles more numbers, and that the
sums must still be kept in a wider format or small terms get lost; the result is
checked against a reference either way.  The pages give no format, no scaling
rule and no tolerance, so this module fixes them (each reading is listed in the
design notes):

Format.  E4M3 as in the OCP 8-bit floating-point specification, variant without
infinities: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.  Exponent
field 0 holds subnormals m/8 * 2^-6; fields 1..15 hold (1 + m/8) * 2^(e-7),
except S.1111.111 which is NaN.  Largest finite value 448, smallest subnormal
2^-9.  Rounding is to nearest, ties to even, and out-of-range values saturate
to +-448.

Quantisation (per tile).  For every 128-row tile of one head of Q, K or V (rows
are sequence positions; the last tile may be short), amax = the largest |x| in
the tile, computed on the float32 values of the bf16 inputs.  If amax > 0 the
tile's scale is amax / 448 and each element's code is e4m3(x * (448 / amax)),
with the division and the product each rounded to float32 (the decision that
picks a code is taken in float32 on both sides); an all-zero tile has scale 0
and all codes 0.  The value a code stands for is e4m3_value(code) * scale.

Reference.  The FP8 forward is attention on the dequantised Q, K, V: the plain
definition in float64 (``oracle.attn_fwd``) applied to those values.  The
GPU's only other approximation is P rounded to e4m3 before the P V product;
``p_rounding_bound`` gives the per-element bound on what that rounding can
change.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
TILE = 128


def e4m3_round(x):
    """Rounds float32 values to the nearest e4m3 value (ties to even), saturating at +-448.

    Returns float64 values, each exactly representable in e4m3.
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    out = np.zeros_like(a)
    sub = a < 2.0 ** -6
    # subnormal range: a fixed quantum of 2^-9
    out[sub] = np.rint(a[sub] * 2.0 ** 9) * 2.0 ** -9
    norm = ~sub & np.isfinite(a)
    if np.any(norm):
        _, ex = np.frexp(a[norm])          # a = f * 2^ex, f in [0.5, 1)
        quantum = np.ldexp(1.0, ex - 1 - 3)  # 3 mantissa bits below the leading one
        out[norm] = np.rint(a[norm] / quantum) * quantum
    out = np.minimum(out, E4M3_MAX)
    out[np.isinf(a)] = E4M3_MAX
    return np.copysign(out, x)


def e4m3_decode(codes):
    """Value of each e4m3 code (uint8); NaN for the two NaN codes."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def e4m3_encode(values):
    """Code of each e4m3-representable value (as returned by e4m3_round)."""
    v = np.asarray(values, dtype=np.float64)
    a = np.abs(v)
    sign = np.where(np.signbit(v), 0x80, 0).astype(np.int64)
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    code[sub] = np.rint(a[sub] * 2.0 ** 9).astype(np.int64)  # 0..7 (8 would be the first normal)
    norm = ~sub
    if np.any(norm):
        f, ex = np.frexp(a[norm])
        e = ex - 1 + 7
        m = np.rint((f * 2.0 - 1.0) * 8.0).astype(np.int64)
        code[norm] = (e << 3) | m
    back = e4m3_decode((code | sign).astype(np.uint8))
    if not np.array_equal(back, v):
        raise ValueError("e4m3_encode: a value is not representable in e4m3")
    return (code | sign).astype(np.uint8)


def quantize_tiles(x, tile: int = TILE):
    """Per-tile e4m3 quantisation of x [..., S, D] along S.

    Returns (codes uint8 [..., S, D], scales float32 [..., ceil(S / tile)]).
    """
    x = np.asarray(x, dtype=np.float32)
    S = x.shape[-2]
    n_tiles = (S + tile - 1) // tile
    codes = np.zeros(x.shape, dtype=np.uint8)
    scales = np.zeros(x.shape[:-2] + (n_tiles,), dtype=np.float32)
    lead = int(np.prod(x.shape[:-2], dtype=np.int64))
    xf = x.reshape(lead, S, x.shape[-1])
    cf = codes.reshape(lead, S, x.shape[-1])
    sf = scales.reshape(lead, n_tiles)
    for i in range(lead):
        for t in range(n_tiles):
            blk = xf[i, t * tile:(t + 1) * tile]
            amax = np.float32(np.max(np.abs(blk))) if blk.size else np.float32(0)
            if amax > 0:
                inv = np.float32(E4M3_MAX) / amax            # float32 division
                sf[i, t] = amax / np.float32(E4M3_MAX)
                y = blk * inv                                # float32 products
                cf[i, t * tile:(t + 1) * tile] = e4m3_encode(e4m3_round(y))
    return codes, scales


def dequantize(codes, scales, tile: int = TILE):
    """Values of per-tile codes: e4m3_value(code) * scale of its tile (float64)."""
    vals = e4m3_decode(codes)
    S = vals.shape[-2]
    rep = np.repeat(np.asarray(scales, dtype=np.float64), tile, axis=-1)[..., :S]
    return vals * rep[..., None]


def _allowed(q_pos, n_keys, causal, block_mask):
    """keep(i, j) for query positions q_pos and keys 0 .. n_keys - 1."""
    q_pos = np.asarray(q_pos)
    j = np.arange(n_keys)
    if block_mask is not None:
        rp, ci = block_mask["row_ptr"], block_mask["col_idx"]
        bs = int(block_mask.get("block_q", 64))
        listed = np.zeros((len(rp) - 1, (n_keys + bs - 1) // bs), dtype=bool)
        for r in range(len(rp) - 1):
            listed[r, ci[rp[r]:rp[r + 1]]] = True
        allowed = listed[q_pos[:, None] // bs, j[None, :] // bs]
        if int(block_mask.get("causal_in_block", 1)):
            allowed &= j[None, :] <= q_pos[:, None]
        return allowed
    if causal:
        return j[None, :] <= q_pos[:, None]
    return np.ones((len(q_pos), n_keys), dtype=bool)


def p_rounding_bound(q, k, v, v_scales, *, scale, causal=False, block_mask=None, q_pos=None, tile: int = TILE):
    """Per-element bound on |O_gpu - O_ref| from rounding P to e4m3 (float64).

    q [B, Hq, Sq, D] (the query rows at positions q_pos, default 0 .. Sq - 1),
    k, v [B, Hkv, S, D] are the dequantised values and v_scales the V tiles'
    scales.  On the GPU, each key tile j of a KV head is folded into P as
    r_j = s_j / s_ref (s_ref the head's largest V tile scale), and p * r_j is
    rounded to e4m3, where p = exp(s - m_used) with a running maximum m_used at
    most 8 binades below the final maximum.  Rounding changes a value y by at
    most 2^-4 y (normal range) or, below 2^-6, by at most min(y, 2^-10); carried
    to the normalised output that gives, per element,
        |dO_id| <= sum_j (2^-4 P_ij + min(P_ij, 2^-10 / (l_i r_j))) |v_jd|
    with P the exact probabilities and l_i = sum_j exp(s_ij - max_j s_ij).
    Returns (terms, A) where terms is that bound and A = sum_j P_ij |v_jd|.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, Sq, D = q.shape
    S = k.shape[2]
    G = Hq // k.shape[1]
    vs = np.asarray(v_scales, dtype=np.float64)
    allowed = _allowed(np.arange(Sq) if q_pos is None else q_pos, S, causal, block_mask)
    terms = np.zeros_like(q)
    A = np.zeros_like(q)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            s = scale * (q[b, h] @ k[b, g].T)
            s = np.where(allowed, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            m = np.where(np.isfinite(m), m, 0.0)
            e = np.where(allowed, np.exp(s - m), 0.0)
            l = e.sum(axis=1, keepdims=True)
            l = np.where(l > 0, l, 1.0)
            P = e / l
            ref = vs[b, g].max() if vs[b, g].size else 0.0
            r_t = vs[b, g] / ref if ref > 0 else np.ones_like(vs[b, g])
            r = np.repeat(r_t, tile)[:S]
            with np.errstate(divide="ignore"):
                cap = np.where(r > 0, 2.0 ** -10 / (l * r[None, :]), np.inf)
            small = np.where(allowed, np.minimum(P, cap), 0.0)
            av = np.abs(v[b, g])
            A[b, h] = P @ av
            terms[b, h] = (2.0 ** -4) * A[b, h] + small @ av
    return terms, A
