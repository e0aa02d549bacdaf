"""Pins of the oracle's SwiGLU (the MoE down projection's input, DeepSeek-V3
§3.3.3 "low-precision activations" (2)) and of its exact BF16 rounding.

  * silu(g) * up against a 40-digit decimal evaluation (Python's decimal
    exp), independent of numpy;
  * closed forms: silu(0) = 0, silu(-x) = silu(x) - x, silu(x) -> x for
    large x; the gate half is the first half (a planted swap fails);
  * BF16 rounding against a brute-force nearest-even search over the BF16
    bit patterns around each value, ties and the subnormal range included.
"""
from decimal import Decimal, getcontext

import numpy as np

import oracle
from fp8_fine_grained_fp8bs_gb300 import synth


def _silu_decimal(g: float, u: float) -> Decimal:
    getcontext().prec = 40
    G = Decimal(g)
    return G / (Decimal(1) + (-G).exp()) * Decimal(u)


def test_swiglu_vs_decimal():
    rng = np.random.default_rng(3)
    g = np.concatenate([rng.normal(0, 1.7, 60), [0.0, -0.0, 1e-30, -1e-30, 20.0, -20.0, 80.0, -80.0]])
    u = np.concatenate([rng.normal(0, 1.7, 60), [1.0, 2.0, 3.0, -1.0, 0.5, 0.25, -4.0, 8.0]])
    h = np.concatenate([g[:, None], u[:, None]], axis=1).astype(np.float32)
    got = oracle.swiglu(h, 1)[:, 0]
    for gi, ui, v in zip(h[:, 0], h[:, 1], got):
        want = _silu_decimal(float(gi), float(ui))
        if want == 0:
            assert v == 0
        else:
            assert abs(Decimal(float(v)) - want) <= abs(want) * Decimal(2) ** -50


def test_swiglu_closed_forms():
    x = np.linspace(-30, 30, 241).astype(np.float32)
    one = np.ones_like(x)
    s_pos = oracle.swiglu(np.stack([x, one], 1), 1)[:, 0]
    s_neg = oracle.swiglu(np.stack([-x, one], 1), 1)[:, 0]
    assert np.allclose(s_neg, s_pos - x.astype(np.float64), rtol=0, atol=1e-12)
    assert oracle.swiglu(np.array([[0.0, 5.0]], np.float32), 1)[0, 0] == 0.0
    assert abs(oracle.swiglu(np.array([[60.0, 1.0]], np.float32), 1)[0, 0] - 60.0) < 1e-20
    # gate is the first half: swapping the halves changes the result
    h = synth.normal_bf16((4, 256), 1.7, 1, 5)
    a = oracle.swiglu(h, 128)
    b = oracle.swiglu(np.concatenate([h[:, 128:], h[:, :128]], axis=1), 128)
    assert not np.allclose(a, b)


def _bf16_brute(v: float) -> float:
    """Nearest BF16 value (ties to the even pattern) by scanning bit patterns."""
    f = np.float32(v)
    b = int(np.array([f], dtype=np.float32).view(np.uint32)[0]) >> 16
    best, bd = None, None
    for cand in range(max(0, (b & 0x7FFF) - 2), min(0x7F7F, (b & 0x7FFF) + 3)):
        c = float(np.array([(cand | (b & 0x8000)) << 16], dtype=np.uint32).view(np.float32)[0])
        d = abs(c - v)
        if best is None or d < bd or (d == bd and cand % 2 == 0):
            best, bd = c, d
    return best


def test_bf16_rounding_vs_brute_force():
    rng = np.random.default_rng(11)
    vals = list(rng.normal(0, 3, 300)) + list(rng.normal(0, 1e-39, 50))
    # exact ties (midpoints between BF16 neighbours) and their float64 neighbours
    for m in [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 255.5, -2.0 ** -130 * 1.5, 3.0 * 2 ** -134]:
        vals += [m, np.nextafter(m, np.inf), np.nextafter(m, -np.inf)]
    got = oracle.bf16_round_f64(np.array(vals))
    for v, g in zip(vals, got):
        assert float(g) == _bf16_brute(float(v)), v


def test_swiglu_quantize_pipeline_by_hand():
    """The composed oracle (SwiGLU -> BF16 -> 1x128 quantise) on rows worked
    by hand: gate 30 and up 0.5 give v = 30 / (1 + e^-30) * 0.5, which rounds
    to 15 in BF16 (e^-30 is far below half a BF16 ulp of 1), so the group's
    scale is fl32(15 / 448) and every code is +448 (0x7E); negating up flips
    every code to 0xFE; a zero gate row gives scale 0 and zero codes; and
    swapping the gate and up halves (silu(0.5) * 30 = 9.34...) would change
    the scale."""
    inter = 128
    h = np.zeros((3, 2 * inter), np.float32)
    h[0, :inter], h[0, inter:] = 30.0, 0.5
    h[1, :inter], h[1, inter:] = 30.0, -0.5
    h[2, :inter], h[2, inter:] = 0.0, 7.0
    q, s = oracle.swiglu_quantize_1x128(synth.f32_to_bf16_bits(h), inter)
    assert s.shape == (3, 1) and q.shape == (3, inter)
    assert s[0, 0] == np.float32(15.0) / np.float32(448.0)
    assert s[1, 0] == s[0, 0]
    assert np.all(q[0] == 0x7E) and np.all(q[1] == 0xFE)
    assert s[2, 0] == 0 and np.all(q[2] == 0)
    swapped = np.float32(0.5 / (1.0 + np.exp(-0.5)) * 30.0)
    assert s[0, 0] != np.float32(swapped) / np.float32(448.0)
