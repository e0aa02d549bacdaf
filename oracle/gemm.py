"""Block-scaled FP8 GEMM with per-128-K-block dequantisation.

TEST INFRASTRUCTURE ONLY (see the package docstring).

DeepSeek-V3 §3.3.2 "increasing accumulation precision" and the Figure 7
explainer ("Increasing accumulation precision"): along the inner dimension
K, every N_C = 128 elements the tensor-core partial sum is promoted to FP32,
multiplied by the two group scales s_a * s_b and added to the accumulator:

    Y[m,n] = sum_kb  P_kb[m,n] * s_a[m,kb] * s_b(n,kb)
    P_kb[m,n] = sum_{k in block kb} dec(qa[m,k]) * dec(qb[n,k])

Both operands are K-major: A[M,K], B[N,K] (Y = A B^T).  s_b(n,kb) is
  * "block": the 128x128 weight scale Sb[n // 128, kb], or
  * "row":   a per-row 1x128 scale Sb[n, kb] (the Wgrad GEMM, where both
             operands are activations grouped along the token dimension).

P_kb is computed in float64, where it is exact: an E4M3 x E4M3 product has
at most 8 significant bits and lies in [2^-18, 2^17.7], so every partial sum
of 128 such products is a multiple of 2^-18 below 2^25 in magnitude, which
needs at most 43 bits.  Any summation order therefore gives the true value.
(§3.5.2 makes the same point for 32 products: an exact FP32-style sum of
them needs at least 34 bits.)  The scaled blocks are summed in float64 in
ascending kb order.

The oracle also returns ``T[m,n] = sum_k |s_a a_k s_b b_k|``, the magnitude
sum used to bound the error of an FP32-accumulated result.
"""
from __future__ import annotations

import numpy as np

from .e4m3 import e4m3_decode

GROUP = 128


def gemm_block_scaled(qa, sa, qb, sb, sb_kind: str = "block"):
    """Reference Y (float64) and magnitude sum T for A[M,K] codes x B[N,K] codes.

    sa: [M, K/128] float32.  sb: [N/128, K/128] ("block") or [N, K/128] ("row").
    """
    qa = np.asarray(qa, dtype=np.uint8)
    qb = np.asarray(qb, dtype=np.uint8)
    M, K = qa.shape
    N, K2 = qb.shape
    assert K == K2 and K % GROUP == 0
    nkb = K // GROUP
    sa = np.asarray(sa, dtype=np.float32).astype(np.float64)
    sb = np.asarray(sb, dtype=np.float32).astype(np.float64)
    assert sa.shape == (M, nkb)
    if sb_kind == "block":
        assert sb.shape == ((N + GROUP - 1) // GROUP, nkb)
        sb_rows = sb[np.arange(N) // GROUP]                       # [N, nkb]
    elif sb_kind == "row":
        assert sb.shape == (N, nkb)
        sb_rows = sb
    else:
        raise ValueError(sb_kind)
    a = e4m3_decode(qa)
    b = e4m3_decode(qb)
    Y = np.zeros((M, N), dtype=np.float64)
    T = np.zeros((M, N), dtype=np.float64)
    for kb in range(nkb):
        ks = slice(kb * GROUP, (kb + 1) * GROUP)
        ab, bb = a[:, ks], b[:, ks]
        P = ab @ bb.T                                 # exact block sum
        Pabs = np.abs(ab) @ np.abs(bb).T              # exact
        S = sa[:, kb][:, None] * sb_rows[:, kb][None, :]   # exact (24-bit x 24-bit)
        Y += P * S
        T += Pabs * np.abs(S)
    return Y, T


def grouped_gemm_block_scaled(qa, sa, offsets, qb, sb):
    """MoE grouped GEMM: rows [offsets[g], offsets[g+1]) of A use expert g's B.

    qa [M_total, K], sa [M_total, K/128], offsets [G+1], qb [G, N, K],
    sb [G, N/128, K/128].  Rows not covered by any group are left 0.
    """
    offsets = np.asarray(offsets, dtype=np.int64)
    M = qa.shape[0]
    G, N, _ = qb.shape
    Y = np.zeros((M, N), dtype=np.float64)
    T = np.zeros((M, N), dtype=np.float64)
    for g in range(G):
        lo, hi = int(offsets[g]), int(offsets[g + 1])
        if hi > lo:
            Y[lo:hi], T[lo:hi] = gemm_block_scaled(qa[lo:hi], sa[lo:hi], qb[g], sb[g], "block")
    return Y, T


def bf16_round(y) -> np.ndarray:
    """Round float64 values to BF16 (nearest, ties to even) in one step.

    Returns the rounded values as float64.  Magnitudes are assumed inside
    the BF16 normal range (true for every GEMM output here).
    """
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    quantum = np.exp2((ex.astype(np.int64) - 1 - 7).astype(np.float64))
    v = np.rint(a / quantum) * quantum
    return np.where(a > 0, np.copysign(v, y), y)
