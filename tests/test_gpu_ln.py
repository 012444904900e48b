"""GPU parity of the fused residual add + LayerNorm (ln_residual_fwd through the
binding) against the float64 oracle (oracle/ln.py) on seeded inputs.

Tolerances:
  y    bf16: the bf16 bound of every other test (2e-2 + half a bf16 unit in the
       last place of ref, element-wise; rel-L2 1e-2); float32: max-abs 1e-3 (the float32 bar of the attention tests).
  h    the float32 sum rounded once to the I/O type: within half a unit in the
       last place of the exact sum (at most 2^-8 |h| for bf16, with 8 significand
       bits, and 2^-24 |h| for float32), plus 1e-30 for exact zeros.
  mean, rstd (float32): per-vector sums of 8 (4) values merged in a log-depth
       tree: relative error a few tens of float32 epsilons; checked at 1e-5
       relative to the row's scale (|mean| + standard deviation), and 1e-5
       relative for rstd.
"""

import numpy as np
import pytest
import torch

from bwd_flashattention_fwd_sm_gb300 import layernorm_residual
from oracle.ln import ln_residual

from parity_util import compare

pytestmark = pytest.mark.gpu

SHAPES = [(1, 1), (3, 7), (17, 64), (64, 1000), (128, 4096), (33, 4104), (8, 16384), (300, 768), (5, 2049)]


def inputs(rows, cols, dtype, seed, residual=True, affine=True):
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x = (torch.randn(rows, cols, generator=g) * 2 + 0.5).to(dt)
    r = torch.randn(rows, cols, generator=g).to(dt) if residual else None
    gm = (torch.randn(cols, generator=g) * 0.5 + 1) if affine else None
    bt = torch.randn(cols, generator=g) * 0.1 if affine else None
    return x, r, gm, bt


def run_both(x, r, gm, bt, eps=1e-5):
    dev = torch.device("cuda")
    cu = lambda t: None if t is None else t.to(dev)
    y, h, mean, rstd = layernorm_residual(cu(x), cu(r), cu(gm), cu(bt), eps=eps, return_sum=True,
                                          return_stats=True)
    torch.cuda.synchronize()
    got = [t.double().cpu().numpy() for t in (y, h, mean, rstd)]
    ref = ln_residual(x.double().numpy(), None if r is None else r.double().numpy(),
                      None if gm is None else gm.double().numpy(), None if bt is None else bt.double().numpy(), eps)
    return got, ref


def check(got, ref, dtype, name):
    y, h, mean, rstd = got
    ry, rh, rmean, rrstd = ref
    compare(f"y[{name}]", y, ry, dtype)
    half_ulp = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -24
    assert np.all(np.abs(h - rh) <= half_ulp * np.abs(rh) + 1e-30), f"h[{name}]"
    scale = np.abs(rmean) + 1.0 / rrstd
    assert np.all(np.abs(mean - rmean) <= 1e-5 * scale), f"mean[{name}] {np.max(np.abs(mean - rmean) / scale):.2e}"
    assert np.all(np.abs(rstd - rrstd) <= 1e-5 * rrstd), f"rstd[{name}]"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_ln_residual_parity(shape, dtype):
    rows, cols = shape
    got, ref = run_both(*inputs(rows, cols, dtype, seed=rows * 7 + cols))
    check(got, ref, dtype, f"{rows}x{cols}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ln_without_residual_or_affine(dtype):
    got, ref = run_both(*inputs(40, 1536, dtype, seed=3, residual=False, affine=False))
    check(got, ref, dtype, "plain")


def test_ln_constant_rows_give_beta():
    x = torch.full((4, 512), 3.0, dtype=torch.bfloat16)
    bt = torch.linspace(-1, 1, 512)
    got, ref = run_both(x, None, torch.ones(512), bt)
    assert np.array_equal(got[0], torch.tensor(ref[0]).to(torch.bfloat16).double().numpy())


def test_ln_full_size_sampled_rows():
    """16384 tokens x 4096 hidden, bf16 with residual: whole run, 64 seeded rows checked."""
    x, r, gm, bt = inputs(16384, 4096, "bf16", seed=11)
    dev = torch.device("cuda")
    y, h, mean, rstd = layernorm_residual(x.to(dev), r.to(dev), gm.to(dev), bt.to(dev), return_sum=True,
                                          return_stats=True)
    torch.cuda.synchronize()
    idx = np.sort(np.random.default_rng(12).choice(16384, 64, replace=False))
    ti = torch.from_numpy(idx)
    ref = ln_residual(x[ti].double().numpy(), r[ti].double().numpy(), gm.double().numpy(), bt.double().numpy())
    got = [t.cpu()[ti].double().numpy() for t in (y, h, mean, rstd)]
    check(got, ref, "bf16", "16384x4096")


def test_ln_unaligned_affine_and_rows():
    """gamma / beta views 4 bytes off a 16-byte boundary and an odd row stride:
    the kernel takes its element-by-element path and gives the same result."""
    x, r, gm, bt = inputs(24, 1000, "bf16", seed=31)
    dev = torch.device("cuda")
    gbuf = torch.zeros(1001, device=dev)
    bbuf = torch.zeros(1001, device=dev)
    gbuf[1:] = gm.to(dev)
    bbuf[1:] = bt.to(dev)
    g1, b1 = gbuf[1:], bbuf[1:]
    assert g1.data_ptr() % 16 != 0
    y, h = layernorm_residual(x.to(dev), r.to(dev), g1, b1)
    torch.cuda.synchronize()
    ref = ln_residual(x.double().numpy(), r.double().numpy(), gm.double().numpy(), bt.double().numpy())
    compare("y[unaligned]", y.double().cpu().numpy(), ref[0], "bf16")
