"""Pins of the oracle's power-of-two ("rounded") scales and of the backward
re-tiling (dequantise -> transpose -> requantise 1x128 -> 128x1).

DeepSeek-V3 "Infrastructure" §3.3.3 "low-precision activations" (1): the
activations that the backward pass converts from 1x128 to 128x1 tiles use
scaling factors that are integer powers of two, so that the conversion adds
no quantisation error; §3.5.2 "support for transposed GEMM operations"
describes the conversion itself.  The scale is read as the smallest power of
two 2^k with absmax / 2^k <= 448.

Pins, none of which re-types the oracle's formula:
  * the scale against a brute-force search over k with exact rationals;
  * every code of a power-of-two group against an exact-rational pipeline
    (value / 2^k exactly, nearest E4M3 value by search, ties to even);
  * the property the pages state: with power-of-two scales the re-tiling
    is lossless for values that stay in the E4M3 normal range, i.e. the
    requantised tensor dequantises to exactly the same numbers;
  * a tiny re-tiling worked by hand in rationals (dequantise exactly,
    column absmax, brute-force scale and codes);
  * planted mistakes (floor instead of ceil, no transpose) fail the pins.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle.e4m3 import e4m3_all_finite_values, e4m3_decode
from fp8_fine_grained_fp8bs_gb300 import synth

_E4M3_VALS = [Fraction(float(v)) for v in e4m3_all_finite_values()]


def _brute_pow2(a: Fraction) -> Fraction:
    """Smallest 2^k (k >= -149) with a / 2^k <= 448, by walking k."""
    if a == 0:
        return Fraction(0)
    k = -149
    while Fraction(448) * Fraction(2) ** k < a:
        k += 1
    return Fraction(2) ** k


def _nearest_code(y: Fraction) -> int:
    """Nearest E4M3 code of a rational (ties to the even code, saturating)."""
    neg = y < 0
    a = min(abs(y), Fraction(448))
    best, best_d = None, None
    for c, v in enumerate(_E4M3_VALS):
        d = abs(a - v)
        if best is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best | (0x80 if neg else 0)


def _bf16_values(seed, n):
    """A spread of BF16 magnitudes across many binades, both signs."""
    rng = np.random.default_rng(seed)
    bits = rng.integers(0x0080, 0x7F7F, n).astype(np.uint16)      # normal BF16, positive
    bits |= (rng.integers(0, 2, n).astype(np.uint16) << 15)
    return bits


@pytest.mark.parametrize("a", [448.0, 449.0, 447.0, 1.0, 0.21875, 0.2197265625, 2.0 ** -133,
                               3.0e38, 1.75 * 2 ** -20, 1.7578125 * 2 ** 10, 0.0])
def test_scale_vs_brute_force_special_values(a):
    s = float(oracle.pow2_scale(np.array([a], dtype=np.float32))[0])
    assert Fraction(s) == _brute_pow2(Fraction(float(np.float32(a))))


def test_scale_vs_brute_force_random_bf16():
    bits = _bf16_values(1, 400) & 0x7FFF
    a = oracle.bf16_bits_to_f32(bits)
    s = oracle.pow2_scale(a)
    for ai, si in zip(a, s):
        assert Fraction(float(si)) == _brute_pow2(Fraction(float(ai)))


def test_absmax_lands_in_top_binades_and_never_saturates():
    x = synth.normal_bf16((64, 1024), 1.0, 3, 1, outliers=True)
    q, s = oracle.quantize_act_1x128(x, pow2=True)
    v = oracle.bf16_bits_to_f32(x).astype(np.float64).reshape(64, 8, 128)
    a = np.abs(v).max(axis=2)
    ratio = a / s.astype(np.float64)
    assert np.all(ratio <= 448.0) and np.all(ratio > 224.0)
    # s is a power of two
    m, _ = np.frexp(s.astype(np.float64))
    assert np.all(m == 0.5)


def test_group_codes_vs_exact_rational_pipeline():
    rng = np.random.default_rng(7)
    for trial in range(6):
        bits = _bf16_values(100 + trial, 128)
        if trial == 5:
            bits[:64] = 0                    # small values next to a large one
        xs = oracle.bf16_bits_to_f32(bits)
        q, s = oracle.quantize_groups(xs[None, :], pow2=True)
        fx = [Fraction(float(v)) for v in xs]
        sp = _brute_pow2(max(abs(v) for v in fx))
        assert Fraction(float(s[0])) == sp
        for v, c in zip(fx, q[0]):
            # x / 2^k is exact here (no float32 underflow for these inputs)
            assert int(c) == _nearest_code(v / sp) or (v == 0 and int(c) in (0x00, 0x80))


def test_zero_group_pow2():
    q, s = oracle.quantize_groups(np.zeros((1, 128), dtype=np.float32), pow2=True)
    assert s[0] == 0 and np.all(q == 0)


def _unit_range_input(M, K, seed):
    """|x| in [1, 2) with random signs: within every 1x128 or 128x1 group the
    values are within a factor 2 of the group maximum."""
    rng = np.random.default_rng(seed)
    mag = rng.uniform(1.0, 2.0, (M, K)).astype(np.float32)
    x = np.where(rng.integers(0, 2, (M, K)) == 1, -mag, mag).astype(np.float32)
    return synth.f32_to_bf16_bits(x)


def test_retiling_with_pow2_scales_is_lossless():
    x = _unit_range_input(256, 384, 11)
    q1, s1 = oracle.quantize_act_1x128(x, pow2=True)
    v1 = oracle.dequantize_1x128(q1, s1)                       # [M, K]
    qt, st = oracle.requant_1x128_to_128x1(q1, s1, pow2=True)   # codes of X^T [K, M], scales [K, M/128]
    vt = e4m3_decode(qt) * np.repeat(st.astype(np.float64), 128, axis=1)
    assert np.array_equal(vt, v1.T.astype(np.float64))


def test_retiling_with_float32_scales_is_not_lossless():
    """Control for the pin above: the same data with absmax/448 scales does
    change values when re-tiled (so the lossless pin has teeth)."""
    x = _unit_range_input(256, 384, 11)
    q1, s1 = oracle.quantize_act_1x128(x, pow2=False)
    v1 = oracle.dequantize_1x128(q1, s1)
    qt, st = oracle.requant_1x128_to_128x1(q1, s1, pow2=False)
    vt = (e4m3_decode(qt) * np.repeat(st.astype(np.float64), 128, axis=1)).astype(np.float32)
    assert not np.array_equal(vt, v1.T)


def test_retiling_tiny_case_by_hand():
    """One 128x128 tile built from a few distinct codes; every output code
    and scale is recomputed in rationals."""
    rng = np.random.default_rng(5)
    codes = rng.choice(np.array([0x00, 0x38, 0x3C, 0xB9, 0x47, 0x50, 0xD4, 0x2A, 0x01], dtype=np.uint8),
                       size=(128, 128))
    scales = np.ldexp(1.0, rng.integers(-12, 4, (128, 1))).astype(np.float32)
    qt, st = oracle.requant_1x128_to_128x1(codes, scales, pow2=True)
    dec = [[Fraction(float(v)) for v in row] for row in e4m3_decode(codes)]
    for col in range(0, 128, 9):
        vals = [dec[r][col] * Fraction(float(scales[r, 0])) for r in range(128)]
        sp = _brute_pow2(max(abs(v) for v in vals))
        assert Fraction(float(st[col, 0])) == sp
        for r in range(128):
            want = 0 if sp == 0 else _nearest_code(vals[r] / sp)
            if vals[r] == 0:
                assert int(qt[col, r]) & 0x7F == 0
            else:
                assert int(qt[col, r]) == want


def test_planted_mistakes_fail():
    # floor instead of ceil: the absmax element saturates for most groups
    x = synth.normal_bf16((8, 1024), 1.0, 2, 1)
    a = np.abs(oracle.bf16_bits_to_f32(x).astype(np.float64)).reshape(-1, 128).max(axis=1)
    k_floor = np.floor(np.log2(a / 448.0))
    assert np.any(a / np.ldexp(1.0, k_floor.astype(np.int64)) > 448.0)
    # requantising without the transpose groups the wrong elements
    xu = _unit_range_input(128, 256, 3)
    q1, s1 = oracle.quantize_act_1x128(xu, pow2=True)
    qt, _ = oracle.requant_1x128_to_128x1(q1, s1, pow2=True)
    wrong, _ = oracle.quantize_act_1x128(oracle.dequantize_1x128(q1, s1), pow2=True)
    assert qt.shape != wrong.shape or not np.array_equal(qt, wrong)
