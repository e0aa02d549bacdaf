"""Pins of the oracle's block-scaled GEMM.

  (i)   brute force: a hand-expanded sum in exact rationals on tiny shapes;
  (ii)  unit scales and small-integer codes reduce to an integer matmul;
  (iii) identity weight blocks return the dequantised activations exactly;
  (iv)  an independent formula: float64 matmul of the dequantised tensors;
  (v)   "row" B scales that repeat a block scale give the "block" result;
  (vi)  the grouped GEMM is the dense GEMM per expert segment; padding rows are 0;
  (vii) planted mistakes (a transposed operand, a shifted K block) fail (i).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle.e4m3 import e4m3_decode, e4m3_encode
from fp8_fine_grained_fp8bs_gb300 import synth


def _rand_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x00          # no NaN codes
    return c


def _rand_scales(rng, shape):
    return (np.abs(rng.standard_normal(shape)) * np.exp2(rng.integers(-12, 4, shape))).astype(np.float32)


def _hand_sum(qa, sa, qb, sb, sb_kind):
    """Y[m][n] = sum over k-blocks of (sum_k a*b) * sa * sb, in exact rationals."""
    M, K = qa.shape
    N = qb.shape[0]
    dec = {c: Fraction(float(e4m3_decode(np.array([c], dtype=np.uint8))[0])) for c in range(256)
           if (c & 0x7F) != 0x7F}
    out = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for kb in range(K // 128):
                p = Fraction(0)
                for k in range(kb * 128, kb * 128 + 128):
                    p += dec[int(qa[m, k])] * dec[int(qb[n, k])]
                sbv = sb[n // 128, kb] if sb_kind == "block" else sb[n, kb]
                tot += p * Fraction(float(sa[m, kb])) * Fraction(float(sbv))
            out[m][n] = tot
    return out


def _check_hand(Y, T, ref, nkb):
    for m in range(len(ref)):
        for n in range(len(ref[0])):
            # the oracle rounds only in the float64 outer sum over k blocks
            bound = Fraction(float(T[m, n])) * Fraction(2 * nkb, 2 ** 52)
            assert abs(Fraction(float(Y[m, n])) - ref[m][n]) <= bound, (m, n)


@pytest.mark.parametrize("M,N,K,kind", [(1, 1, 128, "block"), (2, 2, 256, "block"),
                                        (3, 2, 256, "row"), (2, 130, 128, "block")])
def test_brute_force_hand_sum(M, N, K, kind):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    qa, qb = _rand_codes(rng, (M, K)), _rand_codes(rng, (N, K))
    sa = _rand_scales(rng, (M, K // 128))
    sb = _rand_scales(rng, ((N + 127) // 128 if kind == "block" else N, K // 128))
    Y, T = oracle.gemm_block_scaled(qa, sa, qb, sb, kind)
    _check_hand(Y, T, _hand_sum(qa, sa, qb, sb, kind), K // 128)


def test_integer_matmul_special_case():
    rng = np.random.default_rng(5)
    M, N, K = 8, 256, 384
    ia = rng.integers(-8, 9, size=(M, K))
    ib = rng.integers(-8, 9, size=(N, K))
    qa = e4m3_encode(ia.astype(np.float32))
    qb = e4m3_encode(ib.astype(np.float32))
    assert np.array_equal(e4m3_decode(qa), ia)          # small integers are exact in E4M3
    Y, T = oracle.gemm_block_scaled(qa, np.ones((M, 3), np.float32), qb, np.ones((2, 3), np.float32))
    assert np.array_equal(Y, (ia @ ib.T).astype(np.float64))
    assert np.array_equal(T, (np.abs(ia) @ np.abs(ib).T).astype(np.float64))


def test_identity_weight_blocks():
    rng = np.random.default_rng(6)
    M, K = 5, 256
    qa = _rand_codes(rng, (M, K))
    sa = _rand_scales(rng, (M, 2))
    qb = np.zeros((K, K), np.uint8)
    np.fill_diagonal(qb, 0x38)                             # E4M3 1.0
    Y, _ = oracle.gemm_block_scaled(qa, sa, qb, np.ones((2, 2), np.float32))
    want = e4m3_decode(qa) * np.repeat(sa.astype(np.float64), 128, axis=1)
    assert np.array_equal(Y, want)


def test_dequantised_matmul_formula():
    x = synth.normal_bf16((64, 512), 1.0, 0, 1, outliers=True)
    w = synth.normal_bf16((256, 512), 0.02, 0, 2)
    qa, sa = oracle.quantize_act_1x128(x)
    qb, sb = oracle.quantize_weight_128x128(w)
    Y, T = oracle.gemm_block_scaled(qa, sa, qb, sb)
    A = e4m3_decode(qa) * np.repeat(sa.astype(np.float64), 128, axis=1)
    B = e4m3_decode(qb) * np.repeat(np.repeat(sb.astype(np.float64), 128, axis=0), 128, axis=1)
    assert np.all(np.abs(A @ B.T - Y) <= 1e-12 * T)
    # and the FP8 result approximates the BF16 product (reported, loose)
    Xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    Wf = synth.bf16_bits_to_f32(w).astype(np.float64)
    ref = Xf @ Wf.T
    rel = np.sqrt(np.mean((ref - Y) ** 2) / np.mean(ref ** 2))
    assert rel < 0.1


def test_row_scales_equal_block_scales():
    rng = np.random.default_rng(7)
    qa, qb = _rand_codes(rng, (4, 256)), _rand_codes(rng, (256, 256))
    sa, sb = _rand_scales(rng, (4, 2)), _rand_scales(rng, (2, 2))
    Yb, Tb = oracle.gemm_block_scaled(qa, sa, qb, sb, "block")
    Yr, Tr = oracle.gemm_block_scaled(qa, sa, qb, np.repeat(sb, 128, axis=0), "row")
    assert np.array_equal(Yb, Yr) and np.array_equal(Tb, Tr)


def test_grouped_is_dense_per_segment():
    rng = np.random.default_rng(8)
    offsets = np.array([0, 128, 128, 384], dtype=np.int32)   # the middle expert is empty
    G, N, K = 3, 128, 256
    qa = _rand_codes(rng, (384, K))
    qa[200:256] = 0                                           # padding rows of expert 2
    sa = _rand_scales(rng, (384, 2))
    sa[200:256] = 0
    qb = _rand_codes(rng, (G, N, K))
    sb = _rand_scales(rng, (G, 1, 2))
    Y, T = oracle.grouped_gemm_block_scaled(qa, sa, offsets, qb, sb)
    for g, (lo, hi) in enumerate([(0, 128), (128, 384)]):
        gg = 0 if g == 0 else 2
        Yd, _ = oracle.gemm_block_scaled(qa[lo:hi], sa[lo:hi], qb[gg], sb[gg])
        assert np.array_equal(Y[lo:hi], Yd)
    assert np.all(Y[200:256] == 0)


def test_bf16_round():
    y = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8 + 2 ** -30), 3.0e-5, 0.0])
    got = oracle.bf16_round(y)
    assert got[0] == 1.0 and got[1] == 1.0                 # tie -> even
    assert got[2] == 1.0 + 2 ** -6                           # tie -> even (up)
    assert got[3] == -(1.0 + 2 ** -7)                        # above the tie -> away
    assert got[5] == 0.0
    # agreement with the generator's independent float32 -> BF16 rounding
    # wherever the float64 value is exactly a float32
    rng = np.random.default_rng(9)
    v = rng.standard_normal(100000).astype(np.float32)
    ref = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(v)).astype(np.float64)
    assert np.array_equal(oracle.bf16_round(v.astype(np.float64)), ref)


def test_planted_transposed_operand_fails_hand_sum():
    rng = np.random.default_rng(10)
    qa, qb = _rand_codes(rng, (2, 256)), _rand_codes(rng, (2, 256))
    sa, sb = _rand_scales(rng, (2, 2)), _rand_scales(rng, (1, 2))
    ref = _hand_sum(qa, sa, qb, sb, "block")
    Yw, Tw = oracle.gemm_block_scaled(qb, sa, qa, np.repeat(sb, 2, axis=0)[:1], "block")  # A and B swapped
    with pytest.raises(AssertionError):
        _check_hand(Yw, Tw, ref, 2)


def test_planted_shifted_block_scale_fails_hand_sum():
    rng = np.random.default_rng(11)
    qa, qb = _rand_codes(rng, (2, 256)), _rand_codes(rng, (2, 256))
    sa, sb = _rand_scales(rng, (2, 2)), _rand_scales(rng, (1, 2))
    ref = _hand_sum(qa, sa, qb, sb, "block")
    Yw, Tw = oracle.gemm_block_scaled(qa, sa[:, ::-1].copy(), qb, sb, "block")  # kb index reversed
    with pytest.raises(AssertionError):
        _check_hand(Yw, Tw, ref, 2)
