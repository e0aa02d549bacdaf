"""Power-of-two scales and the FP8 re-tiling on the GPU vs the oracle.

DeepSeek-V3 "Infrastructure" §3.3.3 "low-precision activations" (1):
activations that the backward pass re-tiles from 1x128 to 128x1 use
power-of-two scales; §3.5.2 describes the dequantise -> transpose ->
requantise flow.  Codes and scales must be bit-exact with the oracle.  The
re-tiling inputs are made by the oracle (never by the CUDA path).
"""
import numpy as np
import pytest

import oracle
from fp8_fine_grained_fp8bs_gb300 import synth
from _gpu import require_gpu, to_dev, to_dev_bf16, to_host
from _parity import assert_bytes_equal, assert_scales_equal, check_f32

pytestmark = pytest.mark.gpu


def _edge_rows(K):
    rows = []
    rows.append(np.zeros(K, np.float32))
    rows.append(np.full(K, -0.0, np.float32))
    r = np.zeros(K, np.float32); r[::7] = 1e-39; r[3] = 2e-39; rows.append(r)          # subnormal absmax
    r = np.zeros(K, np.float32); r[::5] = 3e-38; rows.append(r)                        # scale below 2^-127
    r = (np.arange(K, dtype=np.float32) % 128) - 64; r[::128] = 448; rows.append(r)    # s = 1
    r = np.arange(K, dtype=np.float32) % 128; r[::128] = 1.75 * 64; rows.append(r)     # absmax = 1.75 * 2^6
    r = np.arange(K, dtype=np.float32) % 128; r[::128] = 1.7578125 * 64; rows.append(r)
    r = np.full(K, 3.0e38, np.float32); r[1::2] = -1.0; rows.append(r)                 # huge absmax
    return synth.f32_to_bf16_bits(np.stack(rows))


def _check_act_pow2(x_bits, transposed=False):
    torch, fp8bs = require_gpu()
    out = fp8bs.quantize_act(to_dev_bf16(x_bits), transposed=transposed, pow2=True)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_act_1x128(x_bits, pow2=True)
    assert_bytes_equal(to_host(out[0]), q_ref, "1x128 codes")
    assert_scales_equal(to_host(out[1]).T, s_ref, "1x128 scales")
    if transposed:
        qt_ref, st_ref = oracle.quantize_act_128x1(x_bits, pow2=True)
        assert_bytes_equal(to_host(out[2]), qt_ref, "128x1 codes")
        assert_scales_equal(to_host(out[3]).T, st_ref, "128x1 scales")


@pytest.mark.parametrize("M,K", [(128, 512), (1, 128), (130, 256), (4096, 7168)])
def test_act_1x128_pow2(M, K):
    _check_act_pow2(synth.normal_bf16((M, K), 1.0, 21, 1, outliers=True))


def test_act_1x128_pow2_edge_rows():
    _check_act_pow2(_edge_rows(512))


@pytest.mark.parametrize("M,K", [(128, 128), (384, 2048)])
def test_act_dual_pow2(M, K):
    _check_act_pow2(synth.normal_bf16((M, K), 1.0, 22, 1, outliers=True), transposed=True)


def test_act_dual_pow2_edge_rows():
    e = _edge_rows(256)
    x = np.concatenate([e, synth.normal_bf16((128 - e.shape[0], 256), 1.0, 23, 1)])
    _check_act_pow2(x, transposed=True)


@pytest.mark.parametrize("N,K", [(128, 128), (384, 1024)])
def test_weight_pow2(N, K):
    torch, fp8bs = require_gpu()
    bits = synth.normal_bf16((N, K), 0.02, 24, 2)
    w = to_dev_bf16(bits)
    q_ref, s_ref = oracle.quantize_weight_128x128(bits, pow2=True)
    wq, sw = fp8bs.quantize_weight(w, pow2=True)
    assert_bytes_equal(to_host(wq), q_ref, "weight codes")
    assert_scales_equal(to_host(sw), s_ref, "weight scales")
    wq, sw, wq_t, sw_t = fp8bs.quantize_weight(w, transposed=True, pow2=True)
    assert_bytes_equal(to_host(wq), q_ref, "weight codes (with transposed copy)")
    assert_bytes_equal(to_host(wq_t), q_ref.T, "transposed codes")
    assert_scales_equal(to_host(sw_t), s_ref.T, "transposed scales")


def _requant_case(M, K, pow2, seed, edge=False):
    torch, fp8bs = require_gpu()
    x = synth.normal_bf16((M, K), 1.0, seed, 1, outliers=True)
    if edge:
        x[: 8] = _edge_rows(K)
    q1, s1 = oracle.quantize_act_1x128(x, pow2=pow2)
    xq = to_dev(q1)
    sx = to_dev(np.ascontiguousarray(s1.T))                       # kb-major [K/128][M]
    xq_t, sx_t = fp8bs.requant_1x128_to_128x1(xq, sx, pow2=pow2)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_get_device_status() == 0
    qt_ref, st_ref = oracle.requant_1x128_to_128x1(q1, s1, pow2=pow2)
    assert_bytes_equal(to_host(xq_t), qt_ref, "re-tiled codes")
    assert_scales_equal(to_host(sx_t).T, st_ref, "re-tiled scales")
    return q1, s1, to_host(xq_t), to_host(sx_t)


@pytest.mark.parametrize("M,K", [(128, 128), (256, 384), (512, 1024)])
@pytest.mark.parametrize("pow2", [True, False])
def test_requant(M, K, pow2):
    _requant_case(M, K, pow2, 30 + M + K)


@pytest.mark.parametrize("pow2", [True, False])
def test_requant_edge_rows(pow2):
    _requant_case(256, 512, pow2, 31, edge=True)


def test_requant_pow2_is_lossless_on_gpu():
    """|x| in [1, 2): the re-tiled tensor dequantises to the same values."""
    rng = np.random.default_rng(9)
    mag = rng.uniform(1.0, 2.0, (256, 384)).astype(np.float32)
    x = synth.f32_to_bf16_bits(np.where(rng.integers(0, 2, mag.shape) == 1, -mag, mag))
    torch, fp8bs = require_gpu()
    q1, s1 = oracle.quantize_act_1x128(x, pow2=True)
    xq_t, sx_t = fp8bs.requant_1x128_to_128x1(to_dev(q1), to_dev(np.ascontiguousarray(s1.T)), pow2=True)
    vt = oracle.e4m3_decode(to_host(xq_t)) * np.repeat(to_host(sx_t).T.astype(np.float64), 128, axis=1)
    assert np.array_equal(vt, oracle.dequantize_1x128(q1, s1).T.astype(np.float64))


@pytest.mark.parametrize("tensor", ["dY_16384x2048", "X_16384x7168"])
@pytest.mark.parametrize("pow2", [True, False])
def test_requant_full_size_sampled(tensor, pow2):
    """The Wgrad workload's dY[16384, 2048] and the benchmark's X[16384, 7168],
    quantised 1x128 by the oracle and re-tiled at full size (2048 and 7168
    tiles: every CTA of the grid through several); columns sampled for the
    oracle (each column's 128x1 groups are independent of the others)."""
    torch, fp8bs = require_gpu()
    x = synth.wgrad(0)[0] if tensor.startswith("dY") else synth.quantize_input(0)
    K = x.shape[1]
    q1, s1 = oracle.quantize_act_1x128(x, pow2=pow2)
    xq_t, sx_t = fp8bs.requant_1x128_to_128x1(to_dev(q1), to_dev(np.ascontiguousarray(s1.T)), pow2=pow2)
    assert fp8bs.fp8bs_get_device_status() == 0
    xq_t, sx_t = to_host(xq_t), to_host(sx_t)
    cols = np.unique(np.concatenate([np.arange(0, K, 37), [K - 1]]))
    v = oracle.dequantize_1x128(q1, s1)[:, cols]
    qt_ref, st_ref = oracle.quantize_act_128x1(v, pow2=pow2)
    assert_bytes_equal(xq_t[cols], qt_ref, "re-tiled codes (sampled columns)")
    assert_scales_equal(sx_t.T[cols], st_ref, "re-tiled scales (sampled columns)")


def test_wgrad_from_retiled_operands():
    """dW = dY^T X with both operands re-tiled from their 1x128 FP8 copies."""
    torch, fp8bs = require_gpu()
    T_, N, K = 512, 256, 384
    dy = synth.normal_bf16((T_, N), 1.0, 41, 4)
    x = synth.normal_bf16((T_, K), 1.0, 41, 1)
    qdy, sdy = oracle.quantize_act_1x128(dy, pow2=True)
    qx, sx = oracle.quantize_act_1x128(x, pow2=True)
    dyq_t, sdy_t = fp8bs.requant_1x128_to_128x1(to_dev(qdy), to_dev(np.ascontiguousarray(sdy.T)), pow2=True)
    xq_t, sx_t = fp8bs.requant_1x128_to_128x1(to_dev(qx), to_dev(np.ascontiguousarray(sx.T)), pow2=True)
    dw = fp8bs.gemm(dyq_t, sdy_t, xq_t, sx_t, sb_kind=fp8bs.SCALE_ROW1x128, out_dtype=torch.float32)
    qa, sa = oracle.requant_1x128_to_128x1(qdy, sdy, pow2=True)
    qb, sb = oracle.requant_1x128_to_128x1(qx, sx, pow2=True)
    Y, Tm = oracle.gemm_block_scaled(qa, sa, qb, sb, "row")
    check_f32(to_host(dw), Y, Tm, "wgrad from re-tiled operands")
