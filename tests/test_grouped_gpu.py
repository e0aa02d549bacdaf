"""Grouped (MoE) block-scaled FP8 GEMM on the GPU vs the oracle.

Expert segments are contiguous, padded with zero rows to multiples of 128
(the dispatched FP8 activations of §3.3.3 "low-precision communication").
Small cases compare every element, including an empty expert; the full
workload (8192 tokens, top-8 of 32 Zipf-weighted experts, hidden 7168,
expert intermediate 2048: gate/up N=4096, then down K=2048 -> N=7168) is
compared on sampled rows and 128-column blocks of every expert.
"""
import numpy as np
import pytest

import oracle
from fp8_fine_grained_fp8bs_gb300 import synth
from _gpu import require_gpu, to_dev, to_dev_bf16, to_host
from _parity import check_bf16, check_f32

pytestmark = pytest.mark.gpu


def _quantize_weights(fp8bs, w_bits):
    """Quantise every expert's weight on the GPU into one [G,N,K] tensor."""
    import torch
    G, N, K = w_bits.shape
    wq = torch.empty((G, N, K), dtype=torch.uint8, device="cuda:0")
    sw = torch.empty((G, N // 128, K // 128), dtype=torch.float32, device="cuda:0")
    for g in range(G):
        w = to_dev_bf16(w_bits[g])
        fp8bs.fp8bs_quantize_weight(w, N, K, K, wq[g], sw[g])
    return wq, sw


def _run(x_bits, offsets, w_bits, out_bf16, on_device=False):
    torch, fp8bs = require_gpu()
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x_bits))
    wq, sw = _quantize_weights(fp8bs, w_bits)
    out = fp8bs.grouped_gemm(xq, sx, to_dev(offsets.astype(np.int32)), wq, sw,
                             out_dtype=torch.bfloat16 if out_bf16 else torch.float32)
    assert fp8bs.fp8bs_get_device_status() == 0
    return out if on_device else to_host(out)


@pytest.mark.parametrize("out_bf16", [False, True])
def test_small_groups_full_compare(out_bf16):
    G, N, K = 4, 256, 384
    offsets = np.array([0, 128, 128, 384, 512], np.int64)     # expert 1 is empty
    x = synth.normal_bf16((512, K), 1.0, 2, 1, outliers=True)
    x[200:256] = 0                                             # padding rows of expert 2
    x[500:] = 0
    w = synth.normal_bf16((G, N, K), 0.02, 2, 5)
    y = _run(x, offsets, w, out_bf16)
    qa, sa = oracle.quantize_act_1x128(x)
    qb = np.stack([oracle.quantize_weight_128x128(w[g])[0] for g in range(G)])
    sb = np.stack([oracle.quantize_weight_128x128(w[g])[1] for g in range(G)])
    Y, T = oracle.grouped_gemm_block_scaled(qa, sa, offsets, qb, sb)
    if out_bf16:
        check_bf16(y, Y, T, "grouped bf16")
    else:
        check_f32(y, Y, T, "grouped f32")
    assert np.all(y[200:256] == 0) and np.all(y[500:] == 0)


@pytest.mark.parametrize("N,offsets,rows", [
    (128, [128, 256, 384], 512),         # 128-wide tiles: rows 0..127 and 384.. not in any group
    (256, [128, 384, 512], 768),         # 256-wide tiles on CTA pairs: the second expert's one m-tile
                                         # pairs with rows 512..639, which no group owns
    (256, [0, 384, 384, 640], 768),      # three m-tiles, an empty expert, then two
])
def test_rows_outside_groups_untouched(N, offsets, rows):
    torch, fp8bs = require_gpu()
    offsets = np.array(offsets, np.int32)
    G, K = len(offsets) - 1, 256
    x = synth.normal_bf16((rows, K), 1.0, 3, 1)
    w = synth.normal_bf16((G, N, K), 0.02, 3, 5)
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x))
    wq, sw = _quantize_weights(fp8bs, w)
    out = torch.full((rows, N), 7.0, dtype=torch.float32, device="cuda:0")
    fp8bs.grouped_gemm(xq, sx, to_dev(offsets), wq, sw, out=out)
    assert fp8bs.fp8bs_get_device_status() == 0
    y = to_host(out)
    lo, hi = int(offsets[0]), int(offsets[-1])
    assert np.all(y[:lo] == 7.0) and np.all(y[hi:] == 7.0)
    qa, sa = oracle.quantize_act_1x128(x)
    qb = np.stack([oracle.quantize_weight_128x128(w[g])[0] for g in range(G)])
    sb = np.stack([oracle.quantize_weight_128x128(w[g])[1] for g in range(G)])
    Y, T = oracle.grouped_gemm_block_scaled(qa, sa, offsets, qb, sb)
    check_f32(y[lo:hi], Y[lo:hi], T[lo:hi], "grouped offset segments")


def test_invalid_offsets_reported():
    torch, fp8bs = require_gpu()
    x = torch.zeros((256, 128), dtype=torch.uint8, device="cuda:0")
    s = torch.zeros((1, 256), dtype=torch.float32, device="cuda:0")
    w = torch.zeros((2, 128, 128), dtype=torch.uint8, device="cuda:0")
    sw = torch.zeros((2, 1, 1), dtype=torch.float32, device="cuda:0")
    out = torch.full((256, 128), 3.0, dtype=torch.float32, device="cuda:0")
    for bad in ([0, 100, 256], [0, 256, 128], [0, 128, 384]):   # not a multiple / decreasing / beyond M
        fp8bs.grouped_gemm(x, s, to_dev(np.array(bad, np.int32)), w, sw, out=out)
        assert fp8bs.fp8bs_get_device_status() == 7
        assert np.all(to_host(out) == 3.0)
    assert fp8bs.fp8bs_get_device_status() == 0


def test_moe_full_workload_sampled():
    torch, fp8bs = require_gpu()
    wl = synth.moe_fprop(0)
    offsets, src = wl["offsets"], wl["src"]
    x_rows = synth.gather_rows(wl["x_tok"], src)               # dispatched rows, zero padding
    G = 32
    rng = np.random.default_rng(4)
    # gate/up: [67712, 7168] x [32][4096, 7168]^T -> BF16
    y1 = _run(x_rows, offsets, wl["w_gate_up"], out_bf16=True, on_device=True)
    # down: [67712, 2048] x [32][7168, 2048]^T -> BF16
    y2 = _run(wl["down_in"], offsets, wl["w_down"], out_bf16=True, on_device=True)
    for y, a_bits, w_bits in ((y1, x_rows, wl["w_gate_up"]), (y2, wl["down_in"], wl["w_down"])):
        N = w_bits.shape[1]
        for g in range(G):
            lo, hi = int(offsets[g]), int(offsets[g + 1])
            rows = np.unique(np.concatenate([rng.integers(lo, hi, 3), [lo, hi - 1]]))
            nb = rng.choice(N // 128, 1)
            cols = (nb[:, None] * 128 + np.arange(128)[None, :]).reshape(-1)
            qa, sa = oracle.quantize_act_1x128(a_bits[rows])
            qb, sb = oracle.quantize_weight_128x128(w_bits[g][cols])
            Y, T = oracle.gemm_block_scaled(qa, sa, qb, sb)
            got = to_host(y[torch.as_tensor(rows, device=y.device)][:, int(cols[0]):int(cols[-1]) + 1])
            check_bf16(got, Y, T, f"moe expert {g}")
        pad = torch.as_tensor(np.nonzero(src < 0)[0], device=y.device)
        assert int(torch.count_nonzero(y[pad])) == 0
        # one whole expert, every row (padding included) and every column: the
        # last expert, the smallest under the Zipf routing
        lo, hi = int(offsets[G - 1]), int(offsets[G])
        qa, sa = oracle.quantize_act_1x128(a_bits[lo:hi])
        qb, sb = oracle.quantize_weight_128x128(w_bits[G - 1])
        Y, T = oracle.gemm_block_scaled(qa, sa, qb, sb)
        check_bf16(to_host(y[lo:hi]), Y, T, f"moe expert {G - 1}, whole segment [{lo}, {hi}) x {N}")


def test_grouped_with_power_of_two_activation_scales():
    """The activations dispatched before the MoE up projection carry
    power-of-two scales (§3.3.3 "low-precision communication"); the grouped
    GEMM consumes them like any other float32 scale."""
    torch, fp8bs = require_gpu()
    G, N, K = 3, 256, 512
    offsets = np.array([0, 256, 384, 640], np.int64)
    x = synth.normal_bf16((640, K), 1.0, 9, 1, outliers=True)
    w = synth.normal_bf16((G, N, K), 0.02, 9, 5)
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x), pow2=True)
    wq, sw = _quantize_weights(fp8bs, w)
    y = to_host(fp8bs.grouped_gemm(xq, sx, to_dev(offsets.astype(np.int32)), wq, sw, out_dtype=torch.float32))
    assert fp8bs.fp8bs_get_device_status() == 0
    qa, sa = oracle.quantize_act_1x128(x, pow2=True)
    qb = np.stack([oracle.quantize_weight_128x128(w[g])[0] for g in range(G)])
    sb = np.stack([oracle.quantize_weight_128x128(w[g])[1] for g in range(G)])
    Y, T = oracle.grouped_gemm_block_scaled(qa, sa, offsets, qb, sb)
    check_f32(y, Y, T, "grouped, power-of-two activation scales")
