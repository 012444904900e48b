"""Oracle for the fused residual add + LayerNorm: the plain definition in float64.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``): only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may use it.

Definition followed (lpqz.cn CUDA tutorial, section 5.2, the formula given
before the kernel): per row, mean = sum(x) / cols, var = sum((x - mean)^2) /
cols (the population variance), y = (x - mean) / sqrt(var + eps) * gamma + beta;
section 5.1 puts a residual add in front (h = x + residual), and the LayerNorm
acts on h.  Two plain passes over each row in float64; the tutorial's one-pass
Welford form reaches the same value up to rounding and is the GPU's business.
"""

from __future__ import annotations

import numpy as np


def ln_residual(x, residual=None, gamma=None, beta=None, eps: float = 1e-5):
    """Returns (y, h, mean, rstd) for x [rows, cols] (any float dtype, widened to float64)."""
    x = np.asarray(x, dtype=np.float64)
    h = x + np.asarray(residual, dtype=np.float64) if residual is not None else x.copy()
    rows, cols = h.shape
    g = np.ones(cols) if gamma is None else np.asarray(gamma, dtype=np.float64)
    b = np.zeros(cols) if beta is None else np.asarray(beta, dtype=np.float64)
    mean = np.empty(rows)
    rstd = np.empty(rows)
    y = np.empty_like(h)
    for r in range(rows):
        row = h[r]
        m = row.sum() / cols
        var = ((row - m) ** 2).sum() / cols
        s = 1.0 / np.sqrt(var + eps)
        mean[r], rstd[r] = m, s
        y[r] = (row - m) * s * g + b
    return y, h, mean, rstd
