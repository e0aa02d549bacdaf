"""Pins of the oracle's E4M3 codec against facts that do not come from the codec.

  * the format facts the pages print (tests/golden/e4m3_format.txt);
  * hand-worked codes (tests/golden/e4m3_worked_codes.txt);
  * an independent nearest-value search over the sorted list of all finite
    E4M3 values, with ties broken towards the even code.
"""
import os

import numpy as np
import pytest

import oracle
from oracle.e4m3 import e4m3_decode, e4m3_encode, e4m3_all_finite_values

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()[:2]
                out[k] = v
    return out


def _read_worked(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            rows.append((float(parts[0]), int(parts[1], 16)))
    return rows


def test_printed_format_facts():
    facts = _read_kv("e4m3_format.txt")
    assert int(facts["sign_bits"]) + int(facts["exponent_bits"]) + int(facts["mantissa_bits"]) == int(facts["total_bits"])
    # The decoder's field split must be 1/4/3: scaling the mantissa field by
    # one step changes the value by 2^-mantissa_bits at exponent field 7 (value 1.x).
    m_bits = int(facts["mantissa_bits"])
    one = 0x38
    assert e4m3_decode(np.array([one]))[0] == 1.0
    assert e4m3_decode(np.array([one + 1]))[0] == 1.0 + 2.0 ** -m_bits
    # the sign is the top bit
    assert e4m3_decode(np.array([one | 0x80]))[0] == -1.0
    vals = e4m3_all_finite_values()
    n12 = int(np.count_nonzero((vals > 1.0) & (vals < 2.0)))
    assert n12 == int(facts["values_strictly_between_1_and_2"])


def test_extremes_and_nan():
    vals = e4m3_all_finite_values()
    assert vals.max() == 448.0 == oracle.E4M3_MAX
    assert vals[0x7E] == 448.0
    assert vals[1] == 2.0 ** -9                 # smallest subnormal
    assert vals[8] == 2.0 ** -6                 # smallest normal
    assert np.all(np.diff(vals) > 0)            # codes 0..0x7E are ordered
    nan = e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))
    assert np.all(np.isnan(nan))
    # exactly 254 finite codes, of which 2 are zeros
    all_vals = e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.count_nonzero(np.isfinite(all_vals)) == 254


def test_worked_codes():
    for v, code in _read_worked("e4m3_worked_codes.txt"):
        got = int(e4m3_encode(np.array([v], dtype=np.float32))[0])
        assert got == code, (v, hex(got), hex(code))


def test_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    back = e4m3_encode(e4m3_decode(codes).astype(np.float32))
    assert np.array_equal(back, codes)


def _brute_force_encode(y):
    """Nearest finite E4M3 value by search; ties to the even code; saturating."""
    y = np.asarray(y, dtype=np.float32)
    vals = e4m3_all_finite_values()                      # 127 ascending values
    a = np.abs(y.astype(np.float64))
    a_c = np.minimum(a, 448.0)
    hi = np.clip(np.searchsorted(vals, a_c, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    dlo = np.abs(a_c - vals[lo])
    dhi = np.abs(vals[hi] - a_c)
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    return (pick | np.where(np.signbit(y), 0x80, 0)).astype(np.uint8)


def test_encode_vs_brute_force_ties_and_neighbours():
    vals = e4m3_all_finite_values()
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)  # exact in float32
    assert np.all(mids.astype(np.float64) == (vals[:-1] + vals[1:]) / 2)
    pts = [vals.astype(np.float32), mids,
           np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(-np.inf)),
           np.array([448, 456, 464, 465, 479, 480, 481, 1e4, 3.4e38, 1e-40, 1e-45, 0.0],
                    dtype=np.float32)]
    y = np.concatenate(pts)
    y = np.concatenate([y, -y])
    assert np.array_equal(e4m3_encode(y), _brute_force_encode(y))


def test_encode_vs_brute_force_random_bits():
    rng = np.random.default_rng(123)
    bits = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    y = bits.view(np.float32)
    y = y[np.isfinite(y)]
    assert np.array_equal(e4m3_encode(y), _brute_force_encode(y))


def test_encode_vs_brute_force_dense_range():
    # every float32 with magnitude in [2^-10, 2^-9) (around the smallest
    # subnormal) and a 1/101 slice of [2^-9, 2^9)
    lo = np.float32(2.0 ** -10).view(np.uint32)
    mid = np.float32(2.0 ** -9).view(np.uint32)
    top = np.float32(2.0 ** 9).view(np.uint32)
    bits = np.concatenate([np.arange(lo, mid, dtype=np.uint32),
                           np.arange(mid, top, 101, dtype=np.uint32)])
    y = bits.view(np.float32)
    assert np.array_equal(e4m3_encode(y), _brute_force_encode(y))
    assert np.array_equal(e4m3_encode(-y), _brute_force_encode(-y))


def test_planted_mistake_is_caught():
    """A codec that rounds ties away from zero must fail the tie pins."""
    vals = e4m3_all_finite_values()
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    wrong = _brute_force_encode(np.nextafter(mids, np.float32(np.inf)))  # ties pushed up
    assert not np.array_equal(wrong, e4m3_encode(mids))
