"""Comparison helpers for the GPU parity tests (CUDA path vs oracle).

Tolerances are those the hot path is specified to meet:
  * E4M3 codes and float32 scales: bit-exact;
  * FP32 GEMM outputs: |gpu - Y| <= 1e-5 * T, with Y the oracle value and
    T = sum_k |s_a a_k s_b b_k| (computed by the oracle in float64);
  * BF16 GEMM outputs: within 1 BF16 ulp of the correctly rounded oracle
    value RNE(Y).  Where |Y| < 2^8 * 1e-5 * T an FP32-accumulated result
    cannot resolve BF16 ulps of the cancelled sum; there the FP32 bound plus
    one BF16 ulp of the result is accepted instead, and such elements are
    counted.
"""
from __future__ import annotations

import numpy as np

import oracle

F32_REL = 1e-5


BF16_MIN_SUBNORMAL = 2.0 ** -133


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of the BF16 grid at v: 2^(e - 7) for |v| in [2^e, 2^(e+1)),
    never below the subnormal spacing 2^-133 (which is also the ulp of 0)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    ulp = np.exp2((ex.astype(np.int64) - 1 - 7).astype(np.float64))
    return np.where(a > 0, np.maximum(ulp, BF16_MIN_SUBNORMAL), BF16_MIN_SUBNORMAL)


def check_f32(gpu, Y, T, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - Y)
    bad = err > F32_REL * T
    if np.any(bad):
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} FP32 outputs out of tolerance; first at {tuple(i)}: "
                             f"gpu={gpu[tuple(i)]!r} oracle={Y[tuple(i)]!r} bound={F32_REL * T[tuple(i)]!r}")
    return float((err / np.maximum(T, 1e-300)).max()) if err.size else 0.0


def check_bf16(gpu, Y, T, what=""):
    """Returns the number of elements accepted through the cancellation branch."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = oracle.bf16_round(Y)
    ok_ulp = np.abs(gpu - ref) <= bf16_ulp(ref)
    cancel = np.abs(Y) < 2.0 ** 8 * F32_REL * T
    ok_cancel = cancel & (np.abs(gpu - Y) <= F32_REL * T + bf16_ulp(gpu))
    bad = ~(ok_ulp | ok_cancel)
    if np.any(bad):
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} BF16 outputs out of tolerance; first at {i}: "
                             f"gpu={gpu[i]!r} RNE(oracle)={ref[i]!r} oracle={Y[i]!r} T={T[i]!r}")
    return int((ok_cancel & ~ok_ulp).sum())


def assert_bytes_equal(gpu, ref, what=""):
    gpu = np.asarray(gpu)
    ref = np.asarray(ref)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    if not np.array_equal(gpu, ref):
        d = np.argwhere(gpu != ref)
        i = tuple(d[0])
        raise AssertionError(f"{what}: {len(d)} mismatches; first at {i}: gpu={gpu[i]!r} oracle={ref[i]!r}")


def assert_scales_equal(gpu, ref, what=""):
    g = np.ascontiguousarray(gpu, dtype=np.float32).view(np.uint32)
    r = np.ascontiguousarray(ref, dtype=np.float32).view(np.uint32)
    assert_bytes_equal(g, r, what)
