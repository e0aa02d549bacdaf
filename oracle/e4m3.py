"""E4M3 codec, written from the format's definition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The bit layout is the one tabulated in the mixed-precision notes of the
distributed-training page ("PyTorch 提供的浮点数格式": float8 (e4m3) has
1 sign bit, 4 exponent bits, 3 mantissa bits).  Exponent bias 7; exponent
field 0 holds the subnormals 0.m * 2^-6; codes 0x7F and 0xFF are NaN and
there are no infinities (OCP "FN" variant), so the largest finite value is
1.75 * 2^8 = 448.

Encoding (DeepSeek-V3 §3.3.2 casts the scaled values to FP8; the rounding
is read as round-to-nearest-even with saturation): the exact value of a
float32 input is rounded to the nearest E4M3 value with ties to the even
mantissa; magnitudes at or above 448 give +-448.  The sign is kept, also
for results that round to zero (-0 -> 0x80).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_BIAS = 7
E4M3_MANT_BITS = 3
E4M3_MIN_NORMAL_EXP = 1 - E4M3_BIAS          # -6


def e4m3_decode(codes) -> np.ndarray:
    """Value of every E4M3 code as float64 (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2((e - E4M3_BIAS).astype(np.float64))
    sub = (m / 8.0) * np.exp2(float(E4M3_MIN_NORMAL_EXP))
    v = sign * np.where(e == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


def e4m3_all_finite_values() -> np.ndarray:
    """All non-negative finite E4M3 values, ascending (codes 0x00..0x7E)."""
    return e4m3_decode(np.arange(0x7F, dtype=np.uint8))


def _binade(a: np.ndarray) -> np.ndarray:
    """floor(log2(a)) for a > 0, exactly (frexp is exact)."""
    _, ex = np.frexp(a)
    return ex.astype(np.int64) - 1


def e4m3_encode(y) -> np.ndarray:
    """Round float32 values to E4M3 codes (nearest-even, saturating).

    NaN inputs are outside the contract (the quantiser never produces them).
    """
    y = np.asarray(y, dtype=np.float32)
    a = np.abs(y.astype(np.float64))                 # exact widening
    neg = np.signbit(y)
    with np.errstate(divide="ignore", invalid="ignore"):
        # Grid spacing of the binade holding a: 2^(e-3) for normals; the
        # subnormal range [0, 2^-6) shares the spacing of binade -6.
        e = np.maximum(np.where(a > 0, _binade(np.where(a > 0, a, 1.0)), E4M3_MIN_NORMAL_EXP),
                       E4M3_MIN_NORMAL_EXP)
        quantum = np.exp2((e - E4M3_MANT_BITS).astype(np.float64))
        n = np.rint(a / quantum)                     # a/quantum is exact; rint: ties to even
        v = n * quantum                              # exact, representable in E4M3 or = 2^(e+1)
    v = np.where(a >= E4M3_MAX, E4M3_MAX, v)
    # Bit pattern of the (exactly representable) magnitude v.
    vb = np.where(v > 0, v, 1.0)
    ev = _binade(vb)
    is_normal = (v >= 2.0 ** E4M3_MIN_NORMAL_EXP)
    mant_norm = np.rint((vb / np.exp2(ev.astype(np.float64)) - 1.0) * 8.0).astype(np.int64)
    exp_norm = ev + E4M3_BIAS
    mant_sub = np.rint(v * 2.0 ** (-(E4M3_MIN_NORMAL_EXP - E4M3_MANT_BITS))).astype(np.int64)
    code = np.where(is_normal, (exp_norm << 3) | mant_norm, mant_sub)
    code = np.where(neg, code | 0x80, code)
    return code.astype(np.uint8)
