"""Quantisation on the GPU vs the oracle: codes and scales bit-exact.

Inputs follow the workloads' recipe (seeded BF16 normals, 0.1% x50
outliers for activations) plus edge cases: ragged M, a single row, all-zero
and negative-zero groups, subnormal-range values, exact E4M3 ties after the
division, and the largest BF16 magnitudes.
"""
import numpy as np
import pytest

import oracle
from fp8_fine_grained_fp8bs_gb300 import synth
from _gpu import require_gpu, to_dev_bf16, to_host
from _parity import assert_bytes_equal, assert_scales_equal

pytestmark = pytest.mark.gpu


def _check_act(x_bits, transposed=False):
    torch, fp8bs = require_gpu()
    x = to_dev_bf16(x_bits)
    out = fp8bs.quantize_act(x, transposed=transposed)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_act_1x128(x_bits)
    assert_bytes_equal(to_host(out[0]), q_ref, "1x128 codes")
    assert_scales_equal(to_host(out[1]).T, s_ref, "1x128 scales (kb-major)")
    if transposed:
        qt_ref, st_ref = oracle.quantize_act_128x1(x_bits)
        assert_bytes_equal(to_host(out[2]), qt_ref, "128x1 codes (transposed)")
        assert_scales_equal(to_host(out[3]).T, st_ref, "128x1 scales (kb-major)")


def _edge_rows(K):
    """Hand-built rows: zero, -0, subnormal-range, ties, huge values."""
    rows = []
    z = np.zeros(K, np.float32)
    rows.append(z.copy())
    rows.append(np.full(K, -0.0, np.float32))
    r = np.zeros(K, np.float32); r[::7] = 1e-38; r[3] = 2e-38; rows.append(r)          # tiny group
    r = np.arange(K, dtype=np.float32) % 128; rows.append(r)                            # absmax 127: near ties
    r = (np.arange(K, dtype=np.float32) % 128) - 64; r[::128] = 448; rows.append(r)    # s = 1: exact ties
    r = np.full(K, 3.0e38, np.float32); r[1::2] = -1.0; rows.append(r)                 # huge absmax
    r = np.zeros(K, np.float32); r[5] = 1e-3; r[6] = 1e-3 * 2 ** -12; rows.append(r)   # subnormal E4M3 codes
    return synth.f32_to_bf16_bits(np.stack(rows))


@pytest.mark.parametrize("M,K", [(128, 512), (1, 128), (3, 384), (130, 256), (257, 7168), (4096, 7168)])
def test_act_1x128_random(M, K):
    _check_act(synth.normal_bf16((M, K), 1.0, 0, 1, outliers=True))


def test_act_1x128_edge_rows():
    K = 512
    e = _edge_rows(K)
    x = np.concatenate([e, synth.normal_bf16((9, K), 1.0, 0, 1, outliers=True)])
    _check_act(x)


def test_act_1x128_strided_input():
    torch, fp8bs = require_gpu()
    bits = synth.normal_bf16((64, 640), 1.0, 3, 1, outliers=True)
    x = to_dev_bf16(bits)[:, :512]                    # ldx = 640 > K = 512
    xq, sx = fp8bs.quantize_act(x)
    q_ref, s_ref = oracle.quantize_act_1x128(np.ascontiguousarray(bits[:, :512]))
    assert_bytes_equal(to_host(xq), q_ref, "codes")
    assert_scales_equal(to_host(sx).T, s_ref, "scales")


@pytest.mark.parametrize("M,K", [(128, 128), (256, 384), (384, 2048)])
def test_act_dual_random(M, K):
    _check_act(synth.normal_bf16((M, K), 1.0, 0, 1, outliers=True), transposed=True)


def test_act_dual_edge_rows():
    K = 384
    e = _edge_rows(K)
    x = np.concatenate([e, synth.normal_bf16((256 - e.shape[0], K), 1.0, 1, 1, outliers=True)])
    _check_act(x, transposed=True)
    _check_act(np.ascontiguousarray(x[::-1]), transposed=True)


def test_act_dual_edge_columns():
    """The hand-built groups as 128x1 column groups (zero, -0, tiny, ties, huge)."""
    e = _edge_rows(128)
    block = np.concatenate([e, synth.normal_bf16((128 - e.shape[0], 128), 1.0, 1, 3, outliers=True)])
    x = np.ascontiguousarray(np.concatenate([block.T, block[::-1].T], axis=0))   # [256, 128]
    _check_act(x, transposed=True)


@pytest.mark.parametrize("N,K", [(128, 128), (256, 512), (384, 1024)])
def test_weight_random(N, K):
    torch, fp8bs = require_gpu()
    w_bits = synth.normal_bf16((N, K), 0.02, 0, 2)
    w = to_dev_bf16(w_bits)
    wq, sw, wq_t, sw_t = fp8bs.quantize_weight(w, transposed=True)
    q_ref, s_ref = oracle.quantize_weight_128x128(w_bits)
    assert_bytes_equal(to_host(wq), q_ref, "weight codes")
    assert_scales_equal(to_host(sw), s_ref, "weight scales")
    assert_bytes_equal(to_host(wq_t), q_ref.T, "transposed weight codes")
    assert_scales_equal(to_host(sw_t), s_ref.T, "transposed weight scales")
    wq2, sw2 = fp8bs.quantize_weight(w)
    assert_bytes_equal(to_host(wq2), q_ref, "weight codes (no transpose)")


def test_weight_edge_blocks():
    torch, fp8bs = require_gpu()
    w = np.zeros((256, 256), np.float32)
    w[128:, :128] = -0.0
    w[:128, 128:] = np.arange(128 * 128, dtype=np.float32).reshape(128, 128) % 97 - 48
    w[128:, 128:] = 1e-37
    w[200, 200] = 5e-36
    bits = synth.f32_to_bf16_bits(w)
    wq, sw = fp8bs.quantize_weight(to_dev_bf16(bits))
    q_ref, s_ref = oracle.quantize_weight_128x128(bits)
    assert_bytes_equal(to_host(wq), q_ref, "codes")
    assert_scales_equal(to_host(sw), s_ref, "scales")
    wq, sw, wq_t, sw_t = fp8bs.quantize_weight(to_dev_bf16(bits), transposed=True)
    assert_bytes_equal(to_host(wq), q_ref, "codes (with transposed copy)")
    assert_bytes_equal(to_host(wq_t), q_ref.T, "transposed codes")
    assert_scales_equal(to_host(sw_t), s_ref.T, "transposed scales")


def test_empty_inputs_are_no_ops():
    torch, fp8bs = require_gpu()
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda:0")
    xq, sx = fp8bs.quantize_act(x)
    assert xq.shape == (0, 256) and sx.shape == (2, 0)


def test_full_size_standalone_quantize_sampled():
    """X[16384, 7168] as the benchmark quantises it; rows sampled for the oracle."""
    torch, fp8bs = require_gpu()
    bits = synth.quantize_input(0)
    xq, sx = fp8bs.quantize_act(to_dev_bf16(bits))
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, 16384, 97), [16383]]))
    q_ref, s_ref = oracle.quantize_act_1x128(bits[rows])
    assert_bytes_equal(to_host(xq)[rows], q_ref, "codes")
    assert_scales_equal(to_host(sx).T[rows], s_ref, "scales")
    # every non-zero group's absmax element maps to +-448 (property at full size)
    q = to_host(xq).reshape(16384, 56, 128)
    assert np.all(np.any((q == 0x7E) | (q == 0xFE), axis=2))


def test_full_size_dual_quantize_sampled():
    """X[16384, 7168] in both layouts, as the benchmark's dual line quantises
    it: 1x128 groups on sampled rows, 128x1 groups on sampled row blocks
    (each 128-row block's column groups are independent of the others)."""
    torch, fp8bs = require_gpu()
    bits = synth.quantize_input(0)
    xq, sx, xq_t, sx_t = fp8bs.quantize_act(to_dev_bf16(bits), transposed=True)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, 16384, 211), [16383]]))
    q_ref, s_ref = oracle.quantize_act_1x128(bits[rows])
    assert_bytes_equal(to_host(xq)[rows], q_ref, "1x128 codes")
    assert_scales_equal(to_host(sx).T[rows], s_ref, "1x128 scales")
    qt, st = to_host(xq_t), to_host(sx_t)
    for rb in (0, 37, 127):
        qt_ref, st_ref = oracle.quantize_act_128x1(bits[128 * rb:128 * (rb + 1)])
        assert_bytes_equal(qt[:, 128 * rb:128 * (rb + 1)], qt_ref, f"128x1 codes, row block {rb}")
        assert_scales_equal(st[rb][:, None], st_ref, f"128x1 scales, row block {rb}")


def test_full_size_weight_with_transposed_copy_sampled():
    """W[7168, 7168] with the transposed copy (the shape and launch of the
    benchmark's weight line, seeded N(0, 0.02) weights); sampled 128-row
    block rows checked in both layouts."""
    torch, fp8bs = require_gpu()
    w_bits = synth.normal_bf16((7168, 7168), 0.02, 0, 2)
    wq, sw, wq_t, sw_t = fp8bs.quantize_weight(to_dev_bf16(w_bits), transposed=True)
    torch.cuda.synchronize()
    q, s, qt, st = to_host(wq), to_host(sw), to_host(wq_t), to_host(sw_t)
    for nb in (0, 23, 55):
        q_ref, s_ref = oracle.quantize_weight_128x128(w_bits[128 * nb:128 * (nb + 1)])
        assert_bytes_equal(q[128 * nb:128 * (nb + 1)], q_ref, f"codes, block row {nb}")
        assert_scales_equal(s[nb:nb + 1], s_ref, f"scales, block row {nb}")
        assert_bytes_equal(qt[:, 128 * nb:128 * (nb + 1)], q_ref.T, f"transposed codes, block row {nb}")
        assert_scales_equal(st[:, nb:nb + 1], s_ref.T, f"transposed scales, block row {nb}")


def _check_act_weight(x_bits, w_bits, pow2=False, rows=None, nblocks=None):
    """The one-launch quantisation of X (1x128) and W (128x128) against the
    oracle (sampled X rows and W block rows at large sizes)."""
    torch, fp8bs = require_gpu()
    x = to_dev_bf16(x_bits) if x_bits.shape[0] else torch.empty(x_bits.shape, dtype=torch.bfloat16, device="cuda:0")
    w = to_dev_bf16(w_bits) if w_bits.shape[0] else torch.empty(w_bits.shape, dtype=torch.bfloat16, device="cuda:0")
    xq, sx, wq, sw = fp8bs.quantize_act_weight(x, w, pow2=pow2)
    assert fp8bs.fp8bs_get_device_status() == 0
    if x_bits.shape[0]:
        r = np.arange(x_bits.shape[0]) if rows is None else rows
        q_ref, s_ref = oracle.quantize_act_1x128(x_bits[r], pow2=pow2)
        assert_bytes_equal(to_host(xq)[r], q_ref, "X codes")
        assert_scales_equal(to_host(sx).T[r], s_ref, "X scales")
    if w_bits.shape[0]:
        nbs = np.arange(w_bits.shape[0] // 128) if nblocks is None else nblocks
        q, s = to_host(wq), to_host(sw)
        for nb in nbs:
            q_ref, s_ref = oracle.quantize_weight_128x128(w_bits[128 * nb:128 * (nb + 1)], pow2=pow2)
            assert_bytes_equal(q[128 * nb:128 * (nb + 1)], q_ref, f"W codes, block row {nb}")
            assert_scales_equal(s[nb:nb + 1], s_ref, f"W scales, block row {nb}")
    return xq, sx, wq, sw


@pytest.mark.parametrize("M,K,N,Kw", [(128, 512, 256, 512), (3, 384, 128, 256), (257, 256, 384, 1024),
                                      (0, 256, 256, 512), (130, 512, 0, 256)])
@pytest.mark.parametrize("pow2", [False, True])
def test_act_weight_one_launch(M, K, N, Kw, pow2):
    x = synth.normal_bf16((M, K), 1.0, 40 + M, 1, outliers=True)
    w = synth.normal_bf16((N, Kw), 0.02, 40 + N, 2)
    _check_act_weight(x, w, pow2)


def test_act_weight_one_launch_edge_values():
    x = np.concatenate([_edge_rows(384), synth.normal_bf16((121, 384), 1.0, 5, 1, outliers=True)])
    wf = np.zeros((256, 256), np.float32)
    wf[128:, :128] = -0.0
    wf[:128, 128:] = np.arange(128 * 128, dtype=np.float32).reshape(128, 128) % 97 - 48
    wf[128:, 128:] = 1e-37
    _check_act_weight(x, synth.f32_to_bf16_bits(wf))


def test_act_weight_one_launch_step_shape():
    """The benchmark step's operands, X[4096,7168] and W[7168,7168]: sampled
    rows and block rows against the oracle, and every byte identical to the
    two separate quantisations."""
    torch, fp8bs = require_gpu()
    x_bits, w_bits = synth.dense_fprop(0)
    xq, sx, wq, sw = _check_act_weight(x_bits, w_bits, rows=np.arange(0, 4096, 331),
                                       nblocks=np.array([0, 29, 55]))
    xq2, sx2 = fp8bs.quantize_act(to_dev_bf16(x_bits))
    wq2, sw2 = fp8bs.quantize_weight(to_dev_bf16(w_bits))
    assert torch.equal(xq, xq2) and torch.equal(sx, sx2)
    assert torch.equal(wq, wq2) and torch.equal(sw, sw2)
