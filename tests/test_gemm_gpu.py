"""Block-scaled FP8 GEMM on the GPU vs the oracle.

The GPU path quantises on the GPU and multiplies on the GPU; the oracle
quantises the same BF16 inputs on the CPU and computes every 128-K block
exactly.  FP32 outputs must satisfy |gpu - Y| <= 1e-5 * sum_k|s_a a s_b b|;
BF16 outputs must be within 1 BF16 ulp of RNE(Y) (see tests/_parity.py).
Small shapes are compared element by element; the full-size workloads on
sampled rows and 128-column blocks (quantisation groups are local, so the
oracle can compute any sampled output exactly).
"""
import numpy as np
import pytest

import oracle
from fp8_fine_grained_fp8bs_gb300 import synth
from _gpu import require_gpu, to_dev, to_dev_bf16, to_host
from _parity import check_bf16, check_f32

pytestmark = pytest.mark.gpu


def _fprop(x_bits, w_bits, out_bf16, rows=None, nblocks=None):
    torch, fp8bs = require_gpu()
    x, w = to_dev_bf16(x_bits), to_dev_bf16(w_bits)
    xq, sx = fp8bs.quantize_act(x)
    wq, sw = fp8bs.quantize_weight(w)
    y = fp8bs.gemm(xq, sx, wq, sw, out_dtype=torch.bfloat16 if out_bf16 else torch.float32)
    assert fp8bs.fp8bs_get_device_status() == 0
    y = to_host(y)
    rows = np.arange(x_bits.shape[0]) if rows is None else rows
    nblocks = np.arange(w_bits.shape[0] // 128) if nblocks is None else nblocks
    cols = (nblocks[:, None] * 128 + np.arange(128)[None, :]).reshape(-1)
    qa, sa = oracle.quantize_act_1x128(x_bits[rows])
    qb, sb = oracle.quantize_weight_128x128(w_bits[cols])
    Y, T = oracle.gemm_block_scaled(qa, sa, qb, sb)
    got = y[np.ix_(rows, cols)]
    if out_bf16:
        return check_bf16(got, Y, T, "fprop bf16")
    return check_f32(got, Y, T, "fprop f32")


def test_tiny_fprop_f32():
    """X[128,512] x W[256,512]^T, FP32 out (the small workload), every element."""
    x, w = synth.tiny_fprop(0)
    _fprop(x, w, out_bf16=False)


def test_tiny_fprop_bf16():
    x, w = synth.tiny_fprop(0)
    _fprop(x, w, out_bf16=True)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (3, 256, 256), (200, 384, 640), (129, 128, 1024),
                                   (300, 640, 384), (1000, 1152, 512)])
def test_ragged_shapes_f32(M, N, K):
    x = synth.normal_bf16((M, K), 1.0, M + N, 1, outliers=True)
    w = synth.normal_bf16((N, K), 0.02, M + N, 2)
    _fprop(x, w, out_bf16=False)


@pytest.mark.parametrize("M,N,K", [(130, 256, 256), (512, 768, 1024)])
def test_ragged_shapes_bf16(M, N, K):
    x = synth.normal_bf16((M, K), 1.0, 7, 1, outliers=True)
    w = synth.normal_bf16((N, K), 0.02, 7, 2)
    _fprop(x, w, out_bf16=True)


@pytest.mark.parametrize("out", ["f32", "bf16", "f32_accumulate"])
def test_pair_tiles_ragged_rows(out):
    """A shape that takes the 256x256 CTA-pair tiles (31 m-tiles x 5 n-tiles is
    more work units than SMs): an odd number of m-tiles, so the last pair's
    second tile lies wholly past M, and a partial last m-tile whose rows past
    M the store clips; every element compared."""
    torch, fp8bs = require_gpu()
    M, N, K = 3900, 1280, 256
    x = synth.normal_bf16((M, K), 1.0, 21, 1, outliers=True)
    w = synth.normal_bf16((N, K), 0.02, 21, 2)
    if out != "f32_accumulate":
        _fprop(x, w, out_bf16=out == "bf16")
        return
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x))
    wq, sw = fp8bs.quantize_weight(to_dev_bf16(w))
    d0 = np.random.default_rng(1).standard_normal((M, N)).astype(np.float32)
    d = to_dev(d0)
    fp8bs.gemm(xq, sx, wq, sw, out=d, accumulate=True)
    assert fp8bs.fp8bs_get_device_status() == 0
    qa, sa = oracle.quantize_act_1x128(x)
    qb, sb = oracle.quantize_weight_128x128(w)
    Y, T = oracle.gemm_block_scaled(qa, sa, qb, sb)
    got = to_host(d).astype(np.float64)
    assert np.all(np.abs(got - (d0 + Y)) <= 1e-5 * T + 2.0 ** -23 * np.abs(d0 + Y))


def test_zero_and_padding_rows():
    x = synth.normal_bf16((256, 256), 1.0, 11, 1, outliers=True)
    x[5] = 0
    x[130:] = 0
    w = synth.normal_bf16((256, 256), 0.02, 11, 2)
    torch, fp8bs = require_gpu()
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x))
    wq, sw = fp8bs.quantize_weight(to_dev_bf16(w))
    y = to_host(fp8bs.gemm(xq, sx, wq, sw, out_dtype=torch.float32))
    assert np.all(y[5] == 0) and np.all(y[130:] == 0)
    _fprop(x, w, out_bf16=False)


def test_accumulate_f32():
    torch, fp8bs = require_gpu()
    x = synth.normal_bf16((256, 512), 1.0, 12, 1)
    w = synth.normal_bf16((384, 512), 0.02, 12, 2)
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x))
    wq, sw = fp8bs.quantize_weight(to_dev_bf16(w))
    d0 = np.random.default_rng(0).standard_normal((256, 384)).astype(np.float32)
    d = to_dev(d0)
    fp8bs.gemm(xq, sx, wq, sw, out=d, accumulate=True)
    qa, sa = oracle.quantize_act_1x128(x)
    qb, sb = oracle.quantize_weight_128x128(w)
    Y, T = oracle.gemm_block_scaled(qa, sa, qb, sb)
    # the addition of D adds one float32 rounding of |D + Y|
    got = to_host(d).astype(np.float64)
    assert np.all(np.abs(got - (d0 + Y)) <= 1e-5 * T + 2.0 ** -23 * np.abs(d0 + Y))


def test_exact_answer_block_accumulation():
    """Inputs whose exact result is known: one large product and many small
    ones per 128-K block.  Probes how precisely the tensor core accumulates
    inside a block (the pages measured ~14 bits on Hopper, §3.5.2)."""
    torch, fp8bs = require_gpu()
    M, N, K = 128, 128, 1024
    a = np.full((M, K), 0x08, np.uint8)            # 2^-6
    b = np.full((N, K), 0x08, np.uint8)            # 2^-6  -> products 2^-12
    a[:, ::128] = 0x7E                              # 448
    b[:, ::128] = 0x7E                              # 448^2 = 200704 per block
    sa = np.ones((K // 128, M), np.float32)
    sb = np.ones((N // 128, K // 128), np.float32)
    y = fp8bs.gemm(to_dev(a), to_dev(sa), to_dev(b), to_dev(sb), out_dtype=torch.float32)
    Y, T = oracle.gemm_block_scaled(a, sa.T, b, sb)
    exact = (200704.0 + 127 * 2.0 ** -12) * (K // 128)
    assert np.all(Y == exact)
    got = to_host(y).astype(np.float64)
    rel = np.abs(got - exact).max() / exact
    print(f"max relative error of the exact-answer probe: {rel:.3e}")
    check_f32(got, Y, T, "exact-answer probe")


def test_dgrad_full_size_sampled():
    """dX[4096,2048] = dY[4096,7168] . W[7168,2048]: B is the transposed
    copy of the 128x128-quantised weight; FP32 out."""
    torch, fp8bs = require_gpu()
    dy_bits, w_bits = synth.dgrad(0)
    dyq, sdy = fp8bs.quantize_act(to_dev_bf16(dy_bits))
    wq, sw, wq_t, sw_t = fp8bs.quantize_weight(to_dev_bf16(w_bits), transposed=True)
    dx = fp8bs.gemm(dyq, sdy, wq_t, sw_t, out_dtype=torch.float32)
    assert fp8bs.fp8bs_get_device_status() == 0
    dx = to_host(dx)
    rows = np.unique(np.concatenate([np.arange(0, 4096, 61), [4095]]))
    qa, sa = oracle.quantize_act_1x128(dy_bits[rows])
    qw, sw_ref = oracle.quantize_weight_128x128(w_bits)
    Y, T = oracle.gemm_block_scaled(qa, sa, np.ascontiguousarray(qw.T), np.ascontiguousarray(sw_ref.T))
    check_f32(dx[rows], Y, T, "dgrad")


def test_wgrad_small():
    """dW = dY^T X with both operands quantised 128x1 along T (row scales on B)."""
    torch, fp8bs = require_gpu()
    T_, N, K = 512, 256, 384
    dy_bits = synth.normal_bf16((T_, N), 1.0, 5, 4)
    x_bits = synth.normal_bf16((T_, K), 1.0, 5, 1)
    _, _, dyq_t, sdy_t = fp8bs.quantize_act(to_dev_bf16(dy_bits), transposed=True)
    _, _, xq_t, sx_t = fp8bs.quantize_act(to_dev_bf16(x_bits), transposed=True)
    dw = fp8bs.gemm(dyq_t, sdy_t, xq_t, sx_t, sb_kind=fp8bs.SCALE_ROW1x128, out_dtype=torch.float32)
    qa, sa = oracle.quantize_act_128x1(dy_bits)
    qb, sb = oracle.quantize_act_128x1(x_bits)
    Y, Tm = oracle.gemm_block_scaled(qa, sa, qb, sb, "row")
    check_f32(to_host(dw), Y, Tm, "wgrad small")


def test_wgrad_full_size_sampled():
    torch, fp8bs = require_gpu()
    dy_bits, x_bits = synth.wgrad(0)
    _, _, dyq_t, sdy_t = fp8bs.quantize_act(to_dev_bf16(dy_bits), transposed=True)
    _, _, xq_t, sx_t = fp8bs.quantize_act(to_dev_bf16(x_bits), transposed=True)
    dw = fp8bs.gemm(dyq_t, sdy_t, xq_t, sx_t, sb_kind=fp8bs.SCALE_ROW1x128, out_dtype=torch.float32)
    assert fp8bs.fp8bs_get_device_status() == 0
    dw = to_host(dw)
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(2048, 24, replace=False))
    cols = np.sort(rng.choice(7168, 512, replace=False))
    qa, sa = oracle.quantize_act_128x1(dy_bits[:, rows])
    qb, sb = oracle.quantize_act_128x1(x_bits[:, cols])
    Y, Tm = oracle.gemm_block_scaled(qa, sa, qb, sb, "row")
    check_f32(dw[np.ix_(rows, cols)], Y, Tm, "wgrad")


@pytest.mark.parametrize("M, N, K", [(256, 384, 512), (200, 256, 384), (2300, 2176, 256)])
@pytest.mark.parametrize("out", ["f32", "bf16", "f32_accumulate"])
def test_row_scaled_b_ragged(M, N, K, out):
    """Row-scaled B (a scale per column of D and 128-K block, as in Wgrad) on
    the 1-CTA tiles (the first two shapes) and on the CTA-pair tiles (the
    third: 18 x 9 tiles of 128 x 256, the last column of tiles half full),
    with ragged M, every output element compared: FP32, BF16 and FP32 added
    into D."""
    torch, fp8bs = require_gpu()
    a_bits = synth.normal_bf16((M, K), 1.0, 21, 1, outliers=True)
    b_bits = synth.normal_bf16((N, K), 0.5, 21, 2)
    aq, sa = fp8bs.quantize_act(to_dev_bf16(a_bits))
    bq, sb = fp8bs.quantize_act(to_dev_bf16(b_bits))
    qa, sa_ref = oracle.quantize_act_1x128(a_bits)
    qb, sb_ref = oracle.quantize_act_1x128(b_bits)
    Y, T = oracle.gemm_block_scaled(qa, sa_ref, qb, sb_ref, "row")
    if out == "bf16":
        d = fp8bs.gemm(aq, sa, bq, sb, sb_kind=fp8bs.SCALE_ROW1x128, out_dtype=torch.bfloat16)
        assert fp8bs.fp8bs_get_device_status() == 0
        check_bf16(to_host(d), Y, T, "row-scaled bf16")
    elif out == "f32":
        d = fp8bs.gemm(aq, sa, bq, sb, sb_kind=fp8bs.SCALE_ROW1x128, out_dtype=torch.float32)
        assert fp8bs.fp8bs_get_device_status() == 0
        check_f32(to_host(d), Y, T, "row-scaled f32")
    else:
        d0 = np.random.default_rng(M).standard_normal((M, N)).astype(np.float32)
        d = to_dev(d0)
        fp8bs.gemm(aq, sa, bq, sb, sb_kind=fp8bs.SCALE_ROW1x128, out=d, accumulate=True)
        assert fp8bs.fp8bs_get_device_status() == 0
        got = to_host(d).astype(np.float64)
        assert np.all(np.abs(got - (d0 + Y)) <= 1e-5 * T + 2.0 ** -23 * np.abs(d0 + Y))


def test_dense_fprop_full_size_sampled():
    """Y[4096,7168] = X[4096,7168] W[7168,7168]^T in BF16, as benchmarked."""
    x_bits, w_bits = synth.dense_fprop(0)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([rng.choice(4096, 40, replace=False), [0, 127, 128, 4095]]))
    nblocks = np.unique(np.concatenate([rng.choice(56, 6, replace=False), [0, 55]]))
    n_cancel = _fprop(x_bits, w_bits, out_bf16=True, rows=rows, nblocks=nblocks)
    print(f"elements accepted through the cancellation branch: {n_cancel}")


@pytest.mark.slow
def test_dense_fprop_full_output():
    """Every element of Y[4096,7168] (BF16 out) against the oracle, as
    benchmarked: the whole output, not samples.  The oracle runs over row
    chunks of 512 to bound host memory (about 40 s of host time)."""
    torch, fp8bs = require_gpu()
    x_bits, w_bits = synth.dense_fprop(0)
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x_bits))
    wq, sw = fp8bs.quantize_weight(to_dev_bf16(w_bits))
    y = to_host(fp8bs.gemm(xq, sx, wq, sw, out_dtype=torch.bfloat16))
    assert fp8bs.fp8bs_get_device_status() == 0
    qa, sa = oracle.quantize_act_1x128(x_bits)
    qb, sb = oracle.quantize_weight_128x128(w_bits)
    n_cancel = 0
    for r0 in range(0, x_bits.shape[0], 512):
        rs = slice(r0, r0 + 512)
        Y, T = oracle.gemm_block_scaled(qa[rs], sa[rs], qb, sb)
        n_cancel += check_bf16(y[rs], Y, T, f"dense fprop rows {r0}..{r0 + 511}")
    print(f"elements accepted through the cancellation branch: {n_cancel}")


def test_bad_arguments_raise():
    torch, fp8bs = require_gpu()
    a = torch.zeros((128, 200), dtype=torch.uint8, device="cuda:0")
    s = torch.zeros((2, 128), dtype=torch.float32, device="cuda:0")
    with pytest.raises(fp8bs.Fp8bsError) as e:
        fp8bs.fp8bs_gemm(a, s, a, s, 0, s, 0, 128, 128, 200)
    assert e.value.status == 2


def test_bounded_wait_expires_and_context_stays_usable():
    """A wait that nothing completes gives up after its limit, the status word
    reports FP8BS_ERR_TIMEOUT (read once, then cleared), and a GEMM launched
    afterwards runs correctly."""
    torch, fp8bs = require_gpu()
    assert fp8bs.fp8bs_get_device_status() == 0
    fp8bs.fp8bs_selftest_wait_timeout(20000)          # 20 ms
    assert fp8bs.fp8bs_get_device_status() == 6       # FP8BS_ERR_TIMEOUT
    assert fp8bs.fp8bs_get_device_status() == 0       # cleared by the read
    x, w = synth.tiny_fprop(0)
    _fprop(x, w, out_bf16=False)
    assert fp8bs.fp8bs_get_device_status() == 0
