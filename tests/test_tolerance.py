"""The bf16 parity bound's rounding term against PyTorch's own bfloat16 rounding.

half_ulp_bf16(x) must be half the distance between the two bfloat16 neighbours
of x, so that rounding any exact value to bf16 moves it by at most that much,
and no less: a smaller term would fail correct results, a larger one would let
wrong ones through.
"""

import numpy as np
import torch

from parity_util import TOL_BF16_ABS, half_ulp_bf16


def _bf16_spacing(x):
    """Distance from |x| rounded down to bf16 to the next bf16 number up (from bit patterns)."""
    a = torch.from_numpy(np.abs(x).astype(np.float32))
    bits = a.view(torch.int32) & ~0xFFFF  # truncate: the bf16 number at or below |x|
    lo = bits.view(torch.float32).double()
    hi = (bits + 0x10000).view(torch.float32).double()
    return (hi - lo).numpy()


def test_half_ulp_is_half_the_bf16_spacing():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 4, 20000),
                        [1.0, 2.0, 4.0, 7.99, 8.0, 8.01, 0.5, -3.0, 1e-30]])
    assert np.array_equal(half_ulp_bf16(x), _bf16_spacing(x) / 2)
    assert half_ulp_bf16(np.array([0.0]))[0] == 0.0


def test_rounding_stays_within_half_ulp_and_reaches_it():
    rng = np.random.default_rng(1)
    # float32 values, rounded once to bf16 as the kernels' float32 results are
    x = (rng.standard_normal(200000) * 10.0 ** rng.integers(-3, 3, 200000)).astype(np.float32).astype(np.float64)
    r = torch.from_numpy(x).float().to(torch.bfloat16).double().numpy()
    err = np.abs(r - x)
    assert np.all(err <= half_ulp_bf16(x))
    # midpoints of bf16 neighbours sit exactly half an ulp away from both
    lo = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    mid = lo + half_ulp_bf16(lo) * np.sign(lo)
    keep = np.abs(mid) < np.ldexp(1.0, np.frexp(np.abs(lo))[1])  # same binade
    assert np.allclose(np.abs(torch.from_numpy(mid[keep]).to(torch.bfloat16).double().numpy() - mid[keep]),
                       half_ulp_bf16(mid[keep]))


def test_rounding_term_matters_only_above_eight():
    # below 8 in magnitude half an ulp is at most 2^-6 < 2e-2: the stated bar alone governs
    assert half_ulp_bf16(np.array([7.999]))[0] == 2.0 ** -6 < TOL_BF16_ABS
    assert half_ulp_bf16(np.array([8.0]))[0] == 2.0 ** -5 > TOL_BF16_ABS


def _round_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).float().to(torch.bfloat16).double().numpy()


def _group_rounding_replay(q, k, v, do, scale, group):
    """float64 replay of the rounding a bf16-operand, float32-accumulate backward
    takes on dK and dV, causal: per query head, P rounded to bf16 for P^T dO,
    D = <dO, O> from the bf16-rounded O, dS = P (dP - D) rounded to bf16 for
    dS^T Q; group sums exact; the result rounded to bf16 once.  Returns the
    exact and the replayed dK, dV."""
    Hq, S, _ = q.shape
    keep = np.tril(np.ones((S, S), bool))
    out = {n: np.zeros(k.shape) for n in ("dk", "dv", "dk_r", "dv_r")}
    for h in range(Hq):
        g = h // group
        s = np.where(keep, scale * q[h] @ k[g].T, -np.inf)
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        dp = do[h] @ v[g].T
        ds = p * (dp - (p * dp).sum(1, keepdims=True))
        out["dv"][g] += p.T @ do[h]
        out["dk"][g] += scale * ds.T @ q[h]
        d_rounded = (_round_bf16(p @ v[g]) * do[h]).sum(1, keepdims=True)
        out["dv_r"][g] += _round_bf16(p).T @ do[h]
        out["dk_r"][g] += scale * _round_bf16(p * (dp - d_rounded)).T @ q[h]
    return {n: (out[n], _round_bf16(out[n + "_r"])) for n in ("dk", "dv")}


def test_group_scaling_of_the_gradient_bar_against_a_rounding_replay():
    """16 query heads, S = 257, causal, head dim 128: the shape of the GQA test
    cases, with the 16 heads grouped 1, 4 and 16 to a KV head."""
    from bwd_flashattention_fwd_sm_gb300 import workloads as W
    from parity_util import group_scale

    rms, ratio_plain, ratio_scaled = {}, {}, {}
    for group in (1, 4, 16):
        wl = W.Workload("replay", 1, 16, 16 // group, 257, 128, "bf16", "causal", seed=357)
        inp = W.make_inputs(wl)
        q, k, v, do = (inp[n][0].double().numpy() for n in ("q", "k", "v", "do"))
        for n, (exact, replay) in _group_rounding_replay(q, k, v, do, wl.scale, group).items():
            err = np.abs(replay - exact)
            rms[group, n] = float(np.sqrt(np.mean(err ** 2)))
            ratio_plain[group, n] = float(np.max(err / (TOL_BF16_ABS + half_ulp_bf16(exact))))
            ratio_scaled[group, n] = float(np.max(err / (TOL_BF16_ABS * group_scale(group) + half_ulp_bf16(exact))))
    for n in ("dk", "dv"):
        # independent roundings add in quadrature: x4 heads per group -> x2 error
        assert 1.6 < rms[4, n] / rms[1, n] < 2.5 and 1.6 < rms[16, n] / rms[4, n] < 2.5, rms
        assert ratio_plain[4, n] < 1.0  # the configurations' largest group meets the stated bar
        assert ratio_scaled[16, n] < 0.75, ratio_scaled  # the scaled bar holds the replay with room
    # at G = 16 the method's own rounding already breaks the unscaled bar
    assert max(ratio_plain[16, "dk"], ratio_plain[16, "dv"]) > 1.0, ratio_plain
