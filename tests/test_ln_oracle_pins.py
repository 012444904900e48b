"""Pins for the LayerNorm oracle (oracle/ln.py) from what the tutorial's formula
and the mathematics fix: hand-worked values, closed forms and invariants."""

import json
import os

import numpy as np
import pytest

from oracle.ln import ln_residual

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "layernorm_closed_form.json")


def test_golden_closed_forms():
    """Values worked by hand from the formula of the lpqz.cn CUDA tutorial, section 5.2."""
    for c in json.load(open(GOLDEN))["cases"]:
        y, h, mean, rstd = ln_residual(np.array(c["x"], float), None if c["residual"] is None else
                                       np.array(c["residual"], float), c["gamma"], c["beta"], c["eps"])
        np.testing.assert_allclose(mean, c["mean"], rtol=0, atol=1e-15)
        np.testing.assert_allclose(1.0 / rstd ** 2 - c["eps"], c["var"], rtol=0, atol=1e-14)
        np.testing.assert_allclose(y, c["y"], rtol=0, atol=1e-14)


@pytest.mark.parametrize("cols", [2, 7, 64, 1000])
def test_unit_gamma_rows_have_mean_0_and_variance_1(cols):
    x = np.random.default_rng(cols).normal(3.0, 2.0, (5, cols))
    y, *_ = ln_residual(x, eps=0.0)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose((y ** 2).mean(axis=1), 1.0, atol=1e-12)


def test_two_columns_closed_form():
    """[a, b] with eps = 0 normalises to [-1, 1] ordered like a, b."""
    y, *_ = ln_residual(np.array([[2.0, 7.0], [4.0, -1.0]]), eps=0.0)
    np.testing.assert_allclose(y, [[-1.0, 1.0], [1.0, -1.0]], atol=1e-15)


def test_single_column_gives_beta():
    y, *_ = ln_residual(np.array([[3.5], [-2.0]]), gamma=[7.0], beta=[0.25])
    np.testing.assert_array_equal(y, [[0.25], [0.25]])


def test_affine_invariance():
    """LN(a x + c) = LN(x) for a > 0 when eps = 0."""
    x = np.random.default_rng(1).normal(size=(4, 33))
    y0, *_ = ln_residual(x, eps=0.0)
    y1, *_ = ln_residual(3.0 * x - 11.0, eps=0.0)
    np.testing.assert_allclose(y0, y1, atol=1e-12)


def test_residual_is_an_add_before_the_norm():
    rng = np.random.default_rng(2)
    x, r = rng.normal(size=(3, 50)), rng.normal(size=(3, 50))
    g, b = rng.normal(size=50), rng.normal(size=50)
    a = ln_residual(x, r, g, b)
    c = ln_residual(x + r, None, g, b)
    d = ln_residual(r, x, g, b)
    for u, v in ((a, c), (a, d)):
        for s, t in zip(u, v):
            np.testing.assert_allclose(s, t, atol=1e-14)
    np.testing.assert_allclose(a[1], x + r, atol=0)


def test_gamma_beta_are_per_column_affine():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(2, 9))
    g, b = rng.normal(size=9), rng.normal(size=9)
    y0, *_ = ln_residual(x)
    y1, *_ = ln_residual(x, gamma=g, beta=b)
    np.testing.assert_allclose(y1, y0 * g + b, atol=1e-14)


def test_eps_enters_under_the_root():
    """Row [0, 2]: var 1, so y = +-1 / sqrt(1 + eps)."""
    y, *_ = ln_residual(np.array([[0.0, 2.0]]), eps=0.5)
    np.testing.assert_allclose(y, [[-1 / np.sqrt(1.5), 1 / np.sqrt(1.5)]], atol=1e-15)
