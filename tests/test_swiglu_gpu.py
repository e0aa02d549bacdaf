"""Fused SwiGLU -> 1x128 quantisation on the GPU vs the oracle.

The reference is the unfused pipeline (DeepSeek-V3 §3.3.3 "low-precision
activations" (2)): v = BF16(silu(gate) * up), then the 1x128 quantisation of
v.  The kernel evaluates silu(gate) * up in FP32 with a relative error below
2^-16 for every gate, so where the exact value lies within that distance of a BF16
rounding boundary both neighbouring BF16 values are correct.  The check:

  * every group whose 128 values are unambiguous: codes and scale bit-exact
    with the oracle;
  * other groups: the scale is the scale of one of the possible absmax
    values, and, given that scale, each code is the code of one of its
    value's possible BF16 roundings (fl32(b / s) then E4M3, as the oracle).
"""
import numpy as np
import pytest

import oracle
from fp8_fine_grained_fp8bs_gb300 import synth
from _gpu import require_gpu, to_dev_bf16, to_host

pytestmark = pytest.mark.gpu

REL = 2.0 ** -16


def _candidates(h_bits, inter):
    v = oracle.swiglu(h_bits, inter)
    lo = oracle.bf16_round_f64(v - REL * np.abs(v))
    hi = oracle.bf16_round_f64(v + REL * np.abs(v))
    return lo, hi


def _scale(a, pow2):
    return oracle.pow2_scale(a) if pow2 else (np.asarray(a, np.float32) / np.float32(448.0)).astype(np.float32)


def _check(h_bits, inter, q_gpu, s_gpu, pow2):
    """Returns (ambiguous elements, ambiguous groups)."""
    M = h_bits.shape[0]
    G = inter // 128
    lo, hi = _candidates(h_bits, inter)
    amb = lo != hi
    q_ref, s_ref = oracle.quantize_act_1x128(synth.f32_to_bf16_bits(lo), pow2=pow2)
    lo3, hi3, amb3 = (x.reshape(M, G, 128) for x in (lo, hi, amb))
    q3, qr3 = q_gpu.reshape(M, G, 128), q_ref.reshape(M, G, 128)
    clean = ~amb3.any(axis=2)
    assert np.array_equal(q3[clean], qr3[clean]), "codes of unambiguous groups"
    assert np.array_equal(s_gpu[clean].view(np.uint32), s_ref[clean].view(np.uint32)), "scales of unambiguous groups"
    for m, g in zip(*np.nonzero(~clean)):
        a_lo = np.abs(lo3[m, g]).astype(np.float64)
        a_hi = np.abs(hi3[m, g]).astype(np.float64)
        small, large = np.minimum(a_lo, a_hi), np.maximum(a_lo, a_hi)
        # every absmax some choice of roundings attains: a candidate magnitude
        # of some element that is at least every element's smaller candidate
        floor = small.max()
        choices = {float(a) for a in np.concatenate([small, large]) if a >= floor}
        s = np.float32(s_gpu[m, g])
        ok_scales = {float(_scale(np.float32(a), pow2)) for a in choices}
        assert float(s) in ok_scales, (m, g, float(s), ok_scales)
        if s == 0:
            assert np.all(q3[m, g] == 0)
            continue
        c_lo = oracle.e4m3_encode((lo3[m, g].astype(np.float32) / s).astype(np.float32))
        c_hi = oracle.e4m3_encode((hi3[m, g].astype(np.float32) / s).astype(np.float32))
        assert np.all((q3[m, g] == c_lo) | (q3[m, g] == c_hi)), (m, g)
    return int(amb.sum()), int((~clean).sum())


def _run(h_bits, inter, pow2):
    torch, fp8bs = require_gpu()
    q, s = fp8bs.swiglu_quantize(to_dev_bf16(h_bits), pow2=pow2)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_get_device_status() == 0
    return to_host(q), to_host(s).T.copy()


@pytest.mark.parametrize("M,I", [(128, 128), (3, 256), (257, 2048), (1024, 2048), (65, 4096)])
@pytest.mark.parametrize("pow2", [False, True])
def test_swiglu_quantize(M, I, pow2):
    h = synth.normal_bf16((M, 2 * I), 1.7, 50 + M, 5)
    q, s = _run(h, I, pow2)
    n_amb, _ = _check(h, I, q, s, pow2)
    # a +-2^-16 relative interval meets a BF16 rounding boundary for about
    # 2^-7 of the values (BF16 keeps 8 significant bits)
    assert n_amb <= max(16, M * I // 64)


def test_swiglu_quantize_edge_values():
    """Zero rows, +-0, large |gate| (silu -> g and -> 0), tiny products, and
    gates from -64 down to -300 with up values up to 3e38."""
    I = 256
    h = synth.normal_bf16((16, 2 * I), 1.7, 61, 5).view(np.uint16).copy()
    f = oracle.bf16_bits_to_f32(h).copy()
    f[0] = 0.0
    f[1, :I] = -0.0
    f[2, :I] = np.linspace(-80, 80, I, dtype=np.float32)
    f[3, :I] = 60.0
    f[3, I:] = np.linspace(-3, 3, I, dtype=np.float32)
    f[4, I:] = 1e-30
    f[5, :I] = -40.0
    # gates far below zero: silu(g) * u = g u e^g stays a normal number where
    # 1 + e^-g is beyond the one-instruction reciprocal's range
    f[6, :I] = np.linspace(-100, -80, I, dtype=np.float32)
    f[6, I:] = 1e30
    f[7, :I] = np.linspace(-200, -64, I, dtype=np.float32)
    f[7, I:] = 1e35
    f[8, :I] = np.repeat(np.float32([-87.5, -88.0, -90.0, -95.0]), I // 4)    # ordinary up values
    f[9, :I] = np.linspace(-300, -150, I, dtype=np.float32)
    f[9, I:] = 3e38
    f[10, :I] = -64.5
    f[10, I:] = np.linspace(-2e27, 2e27, I, dtype=np.float32)
    h = synth.f32_to_bf16_bits(f)
    for pow2 in (False, True):
        q, s = _run(h, I, pow2)
        _check(h, I, q, s, pow2)


def test_swiglu_quantize_strided_input():
    """h with a leading dimension larger than 2I (a view into a wider buffer)."""
    torch, fp8bs = require_gpu()
    M, I = 130, 384
    wide = synth.normal_bf16((M, 2 * I + 64), 1.7, 62, 5)
    hd = to_dev_bf16(wide)[:, : 2 * I]
    q, s = fp8bs.swiglu_quantize(hd)
    torch.cuda.synchronize()
    _check(np.ascontiguousarray(wide[:, : 2 * I]), I, to_host(q), to_host(s).T.copy(), False)


def test_swiglu_quantize_moe_shape_sampled():
    """The MoE down-projection input shape, [67712, 2048] from a [67712, 4096]
    gate/up output; rows sampled for the oracle."""
    torch, fp8bs = require_gpu()
    M, I = 67712, 2048
    h = synth.normal_bf16((M, 2 * I), 1.7, 7, 5)
    q, s = fp8bs.swiglu_quantize(to_dev_bf16(h))
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, M, 499), [M - 1]]))
    _check(np.ascontiguousarray(h[rows]), I, to_host(q)[rows], to_host(s).T[rows].copy(), False)
