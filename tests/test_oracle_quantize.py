"""Pins of the oracle's quantiser.

  * an independent exact-rational pipeline (Python Fractions) for small
    groups: absmax, s = nearest float32 of absmax/448, y = nearest float32 of
    x/s, code = nearest E4M3 value by search with ties to even;
  * the hand-worked s = 1 group of tests/golden/e4m3_worked_codes.txt;
  * invariants: the absmax element maps to +-448 (code 0x7E / 0xFE); the
    dequantised value lies within half an E4M3 step of the input; sign
    symmetry; power-of-two scaling; weight-block transpose symmetry; the
    128x1 grouping of X is the 1x128 grouping of X^T.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle.e4m3 import e4m3_decode, e4m3_all_finite_values
from fp8_fine_grained_fp8bs_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------- exact pipeline
def _f32_nearest(q: Fraction) -> Fraction:
    """Nearest float32 of a rational (ties to even), by construction."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                       # subnormal spacing below 2^-126
    quantum = Fraction(2) ** (e - 23)
    n = round(a / quantum)                 # Fraction.__round__: ties to even
    return sign * n * quantum


_E4M3_VALS = [Fraction(float(v)) for v in e4m3_all_finite_values()]


def _e4m3_nearest_code(y: Fraction, negative: bool) -> int:
    a = min(abs(y), Fraction(448))
    best, best_d = None, None
    for c, v in enumerate(_E4M3_VALS):
        d = abs(a - v)
        if best is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best | (0x80 if negative else 0)


def _exact_group(xs):
    fx = [Fraction(float(v)) for v in xs]
    a = max(abs(v) for v in fx)
    s = _f32_nearest(a / 448)
    if s == 0:
        return [0] * len(xs), 0.0
    codes = []
    for v, x in zip(fx, xs):
        y = _f32_nearest(v / s)
        codes.append(_e4m3_nearest_code(y, np.signbit(np.float32(x))))
    return codes, float(s)


def _bf16(x):
    return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32)))


@pytest.mark.parametrize("case", range(6))
def test_quantize_vs_exact_rational_pipeline(case):
    rng = np.random.default_rng(1000 + case)
    if case == 0:
        g = np.arange(128, dtype=np.float32)            # absmax 127: many near-ties after division
    elif case == 1:
        g = np.arange(-64, 64, dtype=np.float32) * np.float32(3.0)
    elif case == 2:
        g = rng.standard_normal(128).astype(np.float32)
    elif case == 3:
        g = rng.standard_normal(128).astype(np.float32) * np.float32(1e-3)
        g[17] *= 50
    elif case == 4:                                    # tiny values: subnormal E4M3 codes
        g = rng.standard_normal(128).astype(np.float32)
        g[5] = 3e4
    else:
        g = np.ldexp(rng.standard_normal(128), rng.integers(-30, 30, 128)).astype(np.float32)
    g = _bf16(g)
    codes, s = oracle.quantize_groups(g[None, :])
    want_codes, want_s = _exact_group(g)
    assert np.float32(want_s) == s[0]
    assert codes[0].tolist() == want_codes


def test_near_tie_decided_by_float32_quotient():
    # x = 3 with absmax 128: x / s is close to 10.5, a tie between the E4M3
    # values 10 and 11; the float32 quotient decides which side it falls on.
    g = np.zeros(128, dtype=np.float32)
    g[0], g[1] = 128.0, 3.0
    codes, s = oracle.quantize_groups(g[None, :])
    want, want_s = _exact_group(g)
    assert codes[0].tolist() == want and s[0] == np.float32(want_s)
    y = Fraction(3) / Fraction(float(s[0]))
    assert abs(y - Fraction(21, 2)) < Fraction(1, 1000)     # it is a near-tie


def test_worked_group_with_unit_scale():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_worked_codes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                p = line.split()
                rows.append((float(p[0]), int(p[1], 16)))
    g = np.zeros(128, dtype=np.float32)
    for i, (v, _) in enumerate(rows):
        g[i] = v
    codes, s = oracle.quantize_groups(g[None, :])
    assert s[0] == np.float32(1.0)
    for i, (_, c) in enumerate(rows):
        assert codes[0, i] == c, (i, rows[i], hex(codes[0, i]))


def test_zero_group():
    g = np.zeros((2, 128), dtype=np.float32)
    g[1, :] = -0.0
    codes, s = oracle.quantize_groups(g)
    assert np.all(s == 0) and np.all(codes == 0)


def _random_act(M, K, seed):
    return synth.normal_bf16((M, K), 1.0, seed, 1, outliers=True)


def test_absmax_maps_to_448_and_error_bound():
    x = _random_act(64, 1024, 3)
    q, s = oracle.quantize_act_1x128(x)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64).reshape(64, 8, 128)
    qg = q.reshape(64, 8, 128)
    idx = np.argmax(np.abs(xf), axis=2)
    top = np.take_along_axis(qg, idx[..., None], axis=2)[..., 0]
    assert np.all((top == 0x7E) | (top == 0xFE))
    # dequantised error within half an E4M3 step (relative 2^-4 for normals,
    # absolute 2^-10 * s for the subnormal range), plus float32-quotient slack
    deq = e4m3_decode(qg) * s.astype(np.float64)[..., None]
    ratio = np.abs(xf) / s.astype(np.float64)[..., None]
    err = np.abs(deq - xf)
    normal = ratio >= 2.0 ** -6
    slack = 1 + 2.0 ** -20
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(xf[normal]) * slack)
    sb = np.broadcast_to(s.astype(np.float64)[..., None], xf.shape)
    assert np.all(err[~normal] <= 2.0 ** -10 * sb[~normal] * slack)


def test_sign_symmetry():
    x = _random_act(16, 512, 4)
    q, s = oracle.quantize_act_1x128(x)
    qn, sn = oracle.quantize_act_1x128(x ^ np.uint16(0x8000))
    assert np.array_equal(s, sn)
    assert np.array_equal(qn, q ^ np.uint8(0x80))


@pytest.mark.parametrize("j", [-7, -1, 1, 5])
def test_power_of_two_invariance(j):
    x = synth.bf16_bits_to_f32(_random_act(16, 512, 5))
    q, s = oracle.quantize_act_1x128(x)
    q2, s2 = oracle.quantize_act_1x128(np.ldexp(x, j).astype(np.float32))
    assert np.array_equal(q, q2)
    assert np.array_equal(np.ldexp(s, j).astype(np.float32), s2)


def test_weight_transpose_symmetry():
    w = synth.normal_bf16((256, 384), 0.02, 6, 2)
    q, s = oracle.quantize_weight_128x128(w)
    qt, st = oracle.quantize_weight_128x128(np.ascontiguousarray(w.T))
    assert np.array_equal(qt, q.T)
    assert np.array_equal(st, s.T)


def test_weight_block_is_one_group():
    w = synth.bf16_bits_to_f32(synth.normal_bf16((128, 256), 0.02, 7, 2))
    q, s = oracle.quantize_weight_128x128(w)
    for kb in range(2):
        blk = w[:, kb * 128:(kb + 1) * 128].reshape(1, -1)
        qq, ss = oracle.quantize_groups(blk)
        assert ss[0] == s[0, kb]
        assert np.array_equal(qq.reshape(128, 128), q[:, kb * 128:(kb + 1) * 128])


def test_128x1_is_1x128_of_transpose():
    x = _random_act(256, 384, 8)
    qt, st = oracle.quantize_act_128x1(x)
    assert qt.shape == (384, 256) and st.shape == (384, 2)
    xf = synth.bf16_bits_to_f32(x)
    for c in (0, 77, 383):
        for tb in range(2):
            col = xf[tb * 128:(tb + 1) * 128, c][None, :]
            qq, ss = oracle.quantize_groups(col)
            assert ss[0] == st[c, tb]
            assert np.array_equal(qq[0], qt[c, tb * 128:(tb + 1) * 128])
