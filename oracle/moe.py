"""MoE combine: the weighted sum of each token's expert outputs, in BF16.

TEST INFRASTRUCTURE ONLY (see the package docstring).

DeepSeek-V3 "Infrastructure" §3.3.3, low-precision communication: the
combine after the MoE down-projection stays in BF16.  Each token t has k
routed experts with gate weights w[t][j]; its output is

    out[t] = BF16( sum_j w[t][j] * y_j[t] ),

y_j[t] the BF16 output row of its j-th expert.  The reference value is the
sum in float64 (each product of a float32 weight and a BF16 value is exact
in float64; the float64 sum of k of them is the exact value to within
2^-53 of the magnitude sum) rounded once to BF16; T[t][n] = sum_j |w y| is
the magnitude sum that bounds an FP32-accumulated result.
"""
from __future__ import annotations

import numpy as np

from .gemm import bf16_round


def moe_combine(y, idx, w):
    """y [R, N] float (BF16 values); idx [T, k] int rows of y (< 0: none);
    w [T, k] float32.  Returns (out BF16-rounded float64 [T, N], exact sum
    float64 [T, N], magnitude sum float64 [T, N])."""
    y = np.asarray(y, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    w = np.asarray(w, dtype=np.float32).astype(np.float64)
    T, k = idx.shape
    N = y.shape[1]
    Y = np.zeros((T, N), dtype=np.float64)
    A = np.zeros((T, N), dtype=np.float64)
    for j in range(k):
        ok = idx[:, j] >= 0
        rows = np.where(ok, idx[:, j], 0)
        term = np.where(ok[:, None], w[:, j][:, None] * y[rows], 0.0)
        Y += term
        A += np.abs(term)
    return bf16_round(Y), Y, A
