"""Block-scaled FP8 GEMM with power-of-two scales applied by the tensor core
(fp8bs_gemm_pow2, fp8bs_grouped_gemm_pow2) on the GPU vs the oracle.

The operands are quantised with power-of-two ("rounded") scales, DeepSeek-V3
§3.3.3 (1), on the GPU; the oracle quantises the same BF16 inputs the same
way on the CPU and computes D[m][n] = sum_kb P_kb s_a s_b exactly per
128-K block (oracle.gemm_block_scaled: the definition is the same for any
float32 scales, so nothing in the oracle is specific to this kernel).  The
kernel applies the scales inside the MMA (UE8M0 exponents, §3.5.2's group
scaling in the tensor core) and accumulates all of K in FP32 in tensor
memory, so the tolerance is the FP32 one: |gpu - Y| <= 1e-5 * sum|terms|,
and BF16 outputs within 1 BF16 ulp of RNE(Y).
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
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x_bits), pow2=True)
    wq, sw = fp8bs.quantize_weight(to_dev_bf16(w_bits), pow2=True)
    y = fp8bs.gemm(xq, sx, wq, sw, out_dtype=torch.bfloat16 if out_bf16 else torch.float32, pow2=True)
    assert fp8bs.fp8bs_get_device_status() == 0
    y = to_host(y)
    rows = np.arange(x_bits.shape[0]) if rows is None else rows
    nblocks = np.arange(w_bits.shape[0] // 128) if nblocks is None else nblocks
    cols = (nblocks[:, None] * 128 + np.arange(128)[None, :]).reshape(-1)
    qa, sa = oracle.quantize_act_1x128(x_bits[rows], pow2=True)
    qb, sb = oracle.quantize_weight_128x128(w_bits[cols], pow2=True)
    Y, T = oracle.gemm_block_scaled(qa, sa, qb, sb)
    got = y[np.ix_(rows, cols)]
    if out_bf16:
        return check_bf16(got, Y, T, "pow2 fprop bf16")
    return check_f32(got, Y, T, "pow2 fprop f32")


def test_one_tile_128x128x128():
    x = synth.normal_bf16((128, 128), 1.0, 31, 1, outliers=True)
    w = synth.normal_bf16((128, 128), 0.02, 31, 2)
    _fprop(x, w, out_bf16=False)


def test_tiny_workload_f32():
    x, w = synth.tiny_fprop(0)
    _fprop(x, w, out_bf16=False)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (3, 256, 256), (200, 384, 640), (129, 128, 1024),
                                   (300, 640, 384), (1000, 1152, 512), (256, 256, 896)])
def test_ragged_shapes_f32(M, N, K):
    x = synth.normal_bf16((M, K), 1.0, M + N + 1, 1, outliers=True)
    w = synth.normal_bf16((N, K), 0.02, M + N + 1, 2)
    _fprop(x, w, out_bf16=False)


@pytest.mark.parametrize("M,N,K", [(130, 256, 256), (512, 768, 1024)])
def test_ragged_shapes_bf16(M, N, K):
    x = synth.normal_bf16((M, K), 1.0, 8, 1, outliers=True)
    w = synth.normal_bf16((N, K), 0.02, 8, 2)
    _fprop(x, w, out_bf16=True)


@pytest.mark.parametrize("out", ["f32", "bf16", "f32_accumulate"])
def test_pair_tiles_ragged_rows(out):
    """256x256 CTA-pair tiles, an odd number of m-tiles and a partial last
    m-tile; K = 1664 = 13 k-blocks: scale slots of four k-blocks end in a
    partial slot; every element compared."""
    torch, fp8bs = require_gpu()
    M, N, K = 3900, 1280, 1664
    x = synth.normal_bf16((M, K), 1.0, 22, 1, outliers=True)
    w = synth.normal_bf16((N, K), 0.02, 22, 2)
    if out != "f32_accumulate":
        _fprop(x, w, out_bf16=out == "bf16")
        return
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x), pow2=True)
    wq, sw = fp8bs.quantize_weight(to_dev_bf16(w), pow2=True)
    d0 = np.random.default_rng(2).standard_normal((M, N)).astype(np.float32)
    d = to_dev(d0)
    fp8bs.gemm(xq, sx, wq, sw, out=d, accumulate=True, pow2=True)
    assert fp8bs.fp8bs_get_device_status() == 0
    qa, sa = oracle.quantize_act_1x128(x, pow2=True)
    qb, sb = oracle.quantize_weight_128x128(w, pow2=True)
    Y, T = oracle.gemm_block_scaled(qa, sa, qb, sb)
    got = to_host(d).astype(np.float64)
    assert np.all(np.abs(got - (d0 + Y)) <= 1e-5 * T + 2.0 ** -23 * np.abs(d0 + Y))


def test_zero_groups_and_rows():
    """All-zero groups have scale 0 and zero codes: they contribute nothing."""
    torch, fp8bs = require_gpu()
    x = synth.normal_bf16((256, 512), 1.0, 13, 1, outliers=True)
    x[5] = 0
    x[130:] = 0
    x[7, 128:256] = 0
    w = synth.normal_bf16((256, 512), 0.02, 13, 2)
    w[128:, 256:384] = 0
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x), pow2=True)
    wq, sw = fp8bs.quantize_weight(to_dev_bf16(w), pow2=True)
    y = to_host(fp8bs.gemm(xq, sx, wq, sw, out_dtype=torch.float32, pow2=True))
    assert fp8bs.fp8bs_get_device_status() == 0
    assert np.all(y[5] == 0) and np.all(y[130:] == 0)
    _fprop(x, w, out_bf16=False)


def test_ue8m0_extremes():
    """Scales across the whole UE8M0 range, 2^-127 (a float32 subnormal) to
    2^127: per k-block a centre exponent c, B's block scales 2^(c + d) and
    A's row scales 2^(-c + e) with |d|, |e| <= 8 (clipped to [-127, 127]), so
    every s_a s_b stays within 2^+-16 and D finite; random finite codes
    written directly (not from a quantiser)."""
    torch, fp8bs = require_gpu()
    M, N, K = 256, 256, 1024
    nkb = K // 128
    rng = np.random.default_rng(5)
    sign = lambda shape: (rng.integers(0, 2, shape, dtype=np.uint8) << 7).astype(np.uint8)
    a = rng.integers(0, 0x7F, (M, K), dtype=np.uint8) | sign((M, K))
    b = rng.integers(0, 0x7F, (N, K), dtype=np.uint8) | sign((N, K))
    centre = np.array([-127, 127, -126, 126, -60, 60, 0, 5])
    eb = np.clip(centre[None, :] + rng.integers(-8, 9, (N // 128, nkb)), -127, 127)
    ea = np.clip(-centre[None, :] + rng.integers(-8, 9, (M, nkb)), -127, 127)
    assert ea.min() == -127 and ea.max() == 127 and eb.min() == -127 and eb.max() == 127
    sa = np.ldexp(1.0, ea).astype(np.float32)                 # [M, nkb]; 2^-127 is subnormal
    sb = np.ldexp(1.0, eb).astype(np.float32)                 # [N/128, nkb]
    d = fp8bs.gemm(to_dev(a), to_dev(np.ascontiguousarray(sa.T)), to_dev(b), to_dev(sb), out_dtype=torch.float32,
                   pow2=True)
    assert fp8bs.fp8bs_get_device_status() == 0
    Y, T = oracle.gemm_block_scaled(a, sa, b, sb)
    check_f32(to_host(d), Y, T, "UE8M0 extremes")


@pytest.mark.parametrize("bad", [3.0, -1.0, 2.0 ** -130, 1.5 * 2.0 ** -20])
def test_scale_that_is_not_a_power_of_two_is_reported(bad):
    torch, fp8bs = require_gpu()
    x = synth.normal_bf16((256, 256), 1.0, 14, 1)
    w = synth.normal_bf16((256, 256), 0.02, 14, 2)
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x), pow2=True)
    wq, sw = fp8bs.quantize_weight(to_dev_bf16(w), pow2=True)
    sx[1, 77] = bad
    fp8bs.gemm(xq, sx, wq, sw, out_dtype=torch.float32, pow2=True)
    assert fp8bs.fp8bs_get_device_status() == 7        # FP8BS_ERR_DEVICE_ARG
    assert fp8bs.fp8bs_get_device_status() == 0        # read once
    sw[0, 1] = bad
    sx[1, 77] = 1.0
    fp8bs.gemm(xq, sx, wq, sw, out_dtype=torch.float32, pow2=True)
    assert fp8bs.fp8bs_get_device_status() == 7


def test_agrees_with_the_fold_gemm():
    """The same power-of-two operands through the CUDA-core fold GEMM and the
    tensor-core scaled GEMM: both within tolerance of the oracle, and within
    twice the tolerance of each other."""
    torch, fp8bs = require_gpu()
    x = synth.normal_bf16((640, 2048), 1.0, 15, 1, outliers=True)
    w = synth.normal_bf16((768, 2048), 0.02, 15, 2)
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x), pow2=True)
    wq, sw = fp8bs.quantize_weight(to_dev_bf16(w), pow2=True)
    y_fold = to_host(fp8bs.gemm(xq, sx, wq, sw, out_dtype=torch.float32))
    y_mx = to_host(fp8bs.gemm(xq, sx, wq, sw, out_dtype=torch.float32, pow2=True))
    assert fp8bs.fp8bs_get_device_status() == 0
    qa, sa = oracle.quantize_act_1x128(x, pow2=True)
    qb, sb = oracle.quantize_weight_128x128(w, pow2=True)
    Y, T = oracle.gemm_block_scaled(qa, sa, qb, sb)
    check_f32(y_fold, Y, T, "fold")
    check_f32(y_mx, Y, T, "tensor-core scaled")
    assert np.all(np.abs(y_fold.astype(np.float64) - y_mx) <= 2e-5 * T)


@pytest.mark.parametrize("T_,N,K", [(512, 256, 384), (1024, 384, 1280)])
def test_wgrad_row_scaled_b(T_, N, K):
    """dW = dY^T X with both operands in 128x1 groups along T (row scales on
    B), the backward activations re-tiled from 1x128 FP8 with power-of-two
    scales (§3.5.2's transposed-GEMM support; §3.3.3 (1))."""
    torch, fp8bs = require_gpu()
    dy_bits = synth.normal_bf16((T_, N), 1.0, 6, 4)
    x_bits = synth.normal_bf16((T_, K), 1.0, 6, 1)
    dyq, sdy = fp8bs.quantize_act(to_dev_bf16(dy_bits), pow2=True)
    dyq_t, sdy_t = fp8bs.requant_1x128_to_128x1(dyq, sdy, pow2=True)
    _, _, xq_t, sx_t = fp8bs.quantize_act(to_dev_bf16(x_bits), transposed=True, pow2=True)
    dw = fp8bs.gemm(dyq_t, sdy_t, xq_t, sx_t, sb_kind=fp8bs.SCALE_ROW1x128, out_dtype=torch.float32, pow2=True)
    assert fp8bs.fp8bs_get_device_status() == 0
    qa, sa = oracle.requant_1x128_to_128x1(*oracle.quantize_act_1x128(dy_bits, pow2=True), pow2=True)
    qb, sb = oracle.quantize_act_128x1(x_bits, pow2=True)
    Y, Tm = oracle.gemm_block_scaled(qa, sa, qb, sb, "row")
    check_f32(to_host(dw), Y, Tm, "wgrad pow2")


def _grouped_operands(fp8bs, x_bits, w_bits):
    import torch
    G, N, K = w_bits.shape
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x_bits), pow2=True)
    wq = torch.empty((G, N, K), dtype=torch.uint8, device="cuda:0")
    sw = torch.empty((G, N // 128, K // 128), dtype=torch.float32, device="cuda:0")
    for g in range(G):
        fp8bs.fp8bs_quantize_weight_ex(to_dev_bf16(w_bits[g]), N, K, K, wq[g], sw[g], None, None, fp8bs.SCALE_POW2)
    return xq, sx, wq, sw


def _grouped_oracle(x_bits, offsets, w_bits):
    G = w_bits.shape[0]
    qa, sa = oracle.quantize_act_1x128(x_bits, pow2=True)
    qb = np.stack([oracle.quantize_weight_128x128(w_bits[g], pow2=True)[0] for g in range(G)])
    sb = np.stack([oracle.quantize_weight_128x128(w_bits[g], pow2=True)[1] for g in range(G)])
    return oracle.grouped_gemm_block_scaled(qa, sa, offsets, qb, sb)


@pytest.mark.parametrize("N", [128, 256])
@pytest.mark.parametrize("out_bf16", [False, True])
def test_grouped_small_full_compare(N, out_bf16):
    torch, fp8bs = require_gpu()
    offsets = np.array([0, 128, 128, 512, 640], np.int64)     # an empty expert; 3 m-tiles; 1 m-tile
    x = synth.normal_bf16((768, 384), 1.0, 16, 1, outliers=True)
    x[250:256] = 0
    x[640:] = 0
    w = synth.normal_bf16((4, N, 384), 0.02, 16, 5)
    xq, sx, wq, sw = _grouped_operands(fp8bs, x, w)
    out = torch.full((768, N), 5.0, dtype=torch.bfloat16 if out_bf16 else torch.float32, device="cuda:0")
    fp8bs.grouped_gemm(xq, sx, to_dev(offsets.astype(np.int32)), wq, sw, out=out, pow2=True)
    assert fp8bs.fp8bs_get_device_status() == 0
    y = to_host(out)
    Y, T = _grouped_oracle(x, offsets, w)
    if out_bf16:
        check_bf16(y[:640], Y[:640], T[:640], "grouped pow2 bf16")
    else:
        check_f32(y[:640], Y[:640], T[:640], "grouped pow2 f32")
    assert np.all(y[640:] == 5.0)                              # rows outside every group untouched
    assert np.all(y[250:256] == 0)


def test_grouped_invalid_offsets_reported():
    torch, fp8bs = require_gpu()
    x = torch.zeros((256, 128), dtype=torch.uint8, device="cuda:0")
    s = torch.ones((1, 256), dtype=torch.float32, device="cuda:0")
    w = torch.zeros((2, 256, 128), dtype=torch.uint8, device="cuda:0")
    sw = torch.ones((2, 2, 1), dtype=torch.float32, device="cuda:0")
    out = torch.full((256, 256), 3.0, dtype=torch.float32, device="cuda:0")
    fp8bs.grouped_gemm(x, s, to_dev(np.array([0, 100, 256], np.int32)), w, sw, out=out, pow2=True)
    assert fp8bs.fp8bs_get_device_status() == 7
    assert np.all(to_host(out) == 3.0)


def test_dense_fprop_full_size_sampled():
    """Y[4096,7168] = X[4096,7168] W[7168,7168]^T, BF16 out, both operands
    with power-of-two scales."""
    x_bits, w_bits = synth.dense_fprop(0)
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([rng.choice(4096, 40, replace=False), [0, 127, 128, 255, 256, 4095]]))
    nblocks = np.unique(np.concatenate([rng.choice(56, 6, replace=False), [0, 1, 2, 55]]))
    _fprop(x_bits, w_bits, out_bf16=True, rows=rows, nblocks=nblocks)


def test_moe_full_workload_sampled():
    """The MoE grouped GEMMs (8192 tokens, top-8 of 32 Zipf-weighted experts)
    with power-of-two activation and weight scales; sampled rows and a
    128-column block of every expert, plus the last expert whole."""
    torch, fp8bs = require_gpu()
    wl = synth.moe_fprop(0)
    offsets, src = wl["offsets"], wl["src"]
    x_rows = synth.gather_rows(wl["x_tok"], src)
    G = 32
    rng = np.random.default_rng(6)
    for a_bits, w_bits in ((x_rows, wl["w_gate_up"]), (wl["down_in"], wl["w_down"])):
        N = w_bits.shape[1]
        xq, sx, wq, sw = _grouped_operands(fp8bs, a_bits, w_bits)
        y = fp8bs.grouped_gemm(xq, sx, to_dev(offsets.astype(np.int32)), wq, sw, out_dtype=torch.bfloat16,
                               pow2=True)
        assert fp8bs.fp8bs_get_device_status() == 0
        for g in range(G):
            lo, hi = int(offsets[g]), int(offsets[g + 1])
            rows = np.unique(np.concatenate([rng.integers(lo, hi, 3), [lo, hi - 1]]))
            nb = int(rng.integers(0, N // 128))
            cols = nb * 128 + np.arange(128)
            qa, sa = oracle.quantize_act_1x128(a_bits[rows], pow2=True)
            qb, sb = oracle.quantize_weight_128x128(w_bits[g][cols], pow2=True)
            Y, T = oracle.gemm_block_scaled(qa, sa, qb, sb)
            got = to_host(y[torch.as_tensor(rows, device=y.device)][:, nb * 128:(nb + 1) * 128])
            check_bf16(got, Y, T, f"moe pow2 expert {g}")
        lo, hi = int(offsets[G - 1]), int(offsets[G])
        qa, sa = oracle.quantize_act_1x128(a_bits[lo:hi], pow2=True)
        qb, sb = oracle.quantize_weight_128x128(w_bits[G - 1], pow2=True)
        Y, T = oracle.gemm_block_scaled(qa, sa, qb, sb)
        check_bf16(to_host(y[lo:hi]), Y, T, f"moe pow2 expert {G - 1} whole")
        pad = torch.as_tensor(np.nonzero(src < 0)[0], device=y.device)
        assert int(torch.count_nonzero(y[pad])) == 0
        del xq, sx, wq, sw, y
