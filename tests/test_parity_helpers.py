"""The comparison helpers of the GPU parity tests, checked on the CPU.

The BF16 tolerance is one unit in the last place of the correctly rounded
oracle value; the ulp must follow BF16's grid (8 significant bits, exponent
range of float32, subnormal spacing 2^-133), including at zero, where a
looser ulp would let a wrong non-zero output pass for a zero reference.
"""
import numpy as np
import pytest

from _parity import bf16_ulp, check_bf16, check_f32


@pytest.mark.parametrize("v,ulp", [
    (0.0, 2.0 ** -133), (-0.0, 2.0 ** -133),
    (1.0, 2.0 ** -7), (1.9921875, 2.0 ** -7), (2.0, 2.0 ** -6), (-3.0, 2.0 ** -6),
    (448.0, 2.0), (2.0 ** -126, 2.0 ** -133), (2.0 ** -130, 2.0 ** -133), (3.0e38, 2.0 ** 120),
])
def test_bf16_ulp_values(v, ulp):
    assert float(bf16_ulp(np.array([v]))[0]) == ulp


def test_bf16_check_is_tight_at_zero():
    Y = np.zeros(3)
    T = np.zeros(3)
    assert check_bf16(np.zeros(3), Y, T) == 0
    with pytest.raises(AssertionError):
        check_bf16(np.array([0.0, 0.004, 0.0]), Y, T)          # accepted by an ulp of 2^-7 at zero


def test_bf16_check_one_ulp():
    Y = np.array([1.0 + 2.0 ** -9, 3.0])                      # RNE -> 1.0, 3.0
    T = np.full(2, 1e-3)
    assert check_bf16(np.array([1.0 + 2.0 ** -7, 3.0 - 2.0 ** -6]), Y, T) == 0
    with pytest.raises(AssertionError):
        check_bf16(np.array([1.0 + 2.0 ** -6, 3.0]), Y, T)     # two ulps off


def test_f32_check_bound():
    Y = np.array([1.0, -2.0])
    T = np.array([10.0, 10.0])
    check_f32(Y + 0.9e-4, Y, T)
    with pytest.raises(AssertionError):
        check_f32(Y + np.array([0.0, 1.1e-4]), Y, T)
