"""CPU oracle for the row softmax of "02: Fused softmax" (phobos-lang.dev tutorial).

TEST INFRASTRUCTURE ONLY: used by the tests, the package smoke check and the
benchmark's CPU baseline; never imported by the product path.

What the tutorial's kernel computes, per row i of an [M, pitch] fp32 array of
which the first n columns are the row (tutorial prose and the `softmax`
kernel: mask the columns past n, row maximum, exponentiate the shifted row,
row sum, divide):

    m_i      = max_{j<n} x[i, j]
    y[i, j]  = exp(x[i, j] - m_i) / sum_{k<n} exp(x[i, k] - m_i),   j < n

The kernel gives the columns at or past n the value -1.0e30 so that they
add nothing to the maximum or the sum; here they are simply left out of both
reductions, which is the same thing for every row whose entries exceed
-1.0e30. Columns at or past n are not part of the result.

Everything is evaluated in fp64 from the fp32 inputs (the result is not
rounded to fp32), with numpy's max/exp/sum as the steps; the device result
is compared against it with the tutorial's tolerance, `torch.allclose`'s
defaults (rtol 1e-5, atol 1e-8). IEEE special values follow the definition:
a NaN anywhere in a row, a +inf, or a row of all -inf makes the whole row
NaN; a -inf entry in an otherwise finite row gives 0.
"""
from __future__ import annotations

import numpy as np


def softmax_rows(x: np.ndarray, n: int, rows=None) -> np.ndarray:
    """y[r, j] for the rows `rows` (default: all) and j < n, in fp64.

    x is [M, pitch] with pitch >= n; only x[:, :n] is read.
    """
    x = np.asarray(x)
    if x.ndim != 2 or n < 0 or n > x.shape[1]:
        raise ValueError("x must be 2-D with at least n columns")
    v = x[:, :n] if rows is None else x[np.asarray(rows)][:, :n]
    v = v.astype(np.float64)
    if n == 0:
        return v
    with np.errstate(invalid="ignore", over="ignore"):
        m = v.max(axis=1, keepdims=True)      # NaN-propagating maximum
        e = np.exp(v - m)
        s = e.sum(axis=1, keepdims=True)
        return e / s
