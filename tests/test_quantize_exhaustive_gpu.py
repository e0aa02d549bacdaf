"""Exhaustive pin of the quantisers' division on the GPU.

The kernels never divide per element: each group's scale s and y = RN(1/s)
come from a 128-entry table indexed by the absmax's BF16 mantissa (scaled by
its exponent), and each quotient fl32(x / s) is Markstein's correctly rounded
quotient built from y by two fused multiply-adds; groups whose scale is below
2^-93 take IEEE divisions.  The rule the codes must follow is the plain one
("DeepSeek-V3 FP8 动态量化", "Fine-grained quantization": s = absmax / F_max,
FP8(x) = round(x / s)), as the oracle computes it with IEEE float32 division.

Every quotient that can give a non-zero E4M3 code is covered: for each absmax
mantissa (all 128) at each of 27 absmax exponents from the subnormal range to
the largest finite BF16 binade (spanning the IEEE fallback below biased
exponent 43 and the table path above), one set of groups holds EVERY BF16
value of both signs from the absmax down through 20 binades (quotients from
448 down to about 2^-11.8, below which every code is a signed zero), plus +0
and -0, and the absmax itself with either sign.  Because scaling x and the
absmax by the same power of two scales the exact quotient by 1, this set
reaches every (x mantissa, absmax mantissa, relative binade) combination; the
chosen exponents add the boundaries where the quotient, the scale or the
reciprocal leaves the float32 normal range.  All E4M3 codes, every exact tie
(power-of-two scales) and every near tie are among them.

The same groups go through the 1x128 row path, the 128x1 column path of the
dual-layout kernel, and (one 128x128 block per absmax) the weight paths with
and without the transposed copy, in both scale modes; codes and scales must
be bit-identical to the oracle's.
"""
import numpy as np
import pytest

import oracle
from _gpu import require_gpu, to_dev_bf16, to_host
from _parity import assert_bytes_equal, assert_scales_equal

pytestmark = pytest.mark.gpu

# biased BF16 exponents of the absmax: 0 (subnormal), the IEEE-fallback range
# (< 43), its boundary, the table range, and the top binade
EXPONENTS = [0, 1, 2, 5, 12, 20, 30, 40, 41, 42, 43, 44, 45, 60, 90, 110, 120, 126, 127, 128, 134, 150,
             190, 230, 250, 253, 254]
BINADES_BELOW = 20


def _values_below(a_bits: int) -> np.ndarray:
    """Every BF16 value (both signs) with magnitude in [a * 2^-20, a], plus +0 and -0."""
    lo = max(0, a_bits - BINADES_BELOW * 128)
    pos = np.arange(lo, a_bits + 1, dtype=np.uint16)
    return np.concatenate([pos, pos | np.uint16(0x8000), np.array([0, 0x8000], np.uint16)])


def _groups_for(a_bits: int, flip: bool) -> np.ndarray:
    """Groups of 128 whose absmax is the BF16 value a_bits: element 0 is +-a,
    the other 127 run through _values_below(a_bits) (zero-padded)."""
    v = _values_below(a_bits)
    ng = -(-len(v) // 127)
    body = np.zeros(ng * 127, np.uint16)
    body[: len(v)] = v
    body = body.reshape(ng, 127)
    head = np.full((ng, 1), a_bits, np.uint16)
    if flip:
        head[1::2] |= np.uint16(0x8000)       # absmax element negative in every other group
    return np.concatenate([head, body], axis=1)


def _all_groups(exponents) -> np.ndarray:
    out = []
    for e in exponents:
        for f in range(128):
            a = (e << 7) | f
            if a == 0:
                continue
            out.append(_groups_for(a, flip=(f & 1) == 1))
    return np.concatenate(out)


@pytest.fixture(scope="module")
def groups():
    return _all_groups(EXPONENTS)


@pytest.mark.parametrize("pow2", [False, True])
def test_rows_1x128_every_quotient(groups, pow2):
    torch, fp8bs = require_gpu()
    G = groups.shape[0]
    per_row = 8                                    # K = 1024: eight groups per row
    Gp = -(-G // per_row) * per_row
    g = np.zeros((Gp, 128), np.uint16)
    g[:G] = groups
    x_bits = g.reshape(Gp // per_row, per_row * 128)
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x_bits), pow2=pow2)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_get_device_status() == 0
    q_ref, s_ref = oracle.quantize_act_1x128(x_bits, pow2=pow2)
    assert_bytes_equal(to_host(xq), q_ref, f"1x128 codes (pow2={pow2})")
    assert_scales_equal(to_host(sx).T, s_ref, f"1x128 scales (pow2={pow2})")


@pytest.mark.parametrize("pow2", [False, True])
def test_columns_128x1_every_quotient(groups, pow2):
    """The groups as columns of X[128, G]: the dual kernel's 128x1 output
    quantises exactly these columns (its 1x128 rows mix all groups)."""
    torch, fp8bs = require_gpu()
    G = groups.shape[0]
    Gp = -(-G // 128) * 128
    g = np.zeros((Gp, 128), np.uint16)
    g[:G] = groups
    x_bits = np.ascontiguousarray(g.T)             # [128, Gp]: column j is group j
    xq, sx, xq_t, sx_t = fp8bs.quantize_act(to_dev_bf16(x_bits), transposed=True, pow2=pow2)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_get_device_status() == 0
    qt_ref, st_ref = oracle.quantize_act_128x1(x_bits, pow2=pow2)
    assert_bytes_equal(to_host(xq_t), qt_ref, f"128x1 codes (pow2={pow2})")
    assert_scales_equal(to_host(sx_t).T, st_ref, f"128x1 scales (pow2={pow2})")
    q_ref, s_ref = oracle.quantize_act_1x128(x_bits, pow2=pow2)
    assert_bytes_equal(to_host(xq), q_ref, f"dual kernel 1x128 codes (pow2={pow2})")
    assert_scales_equal(to_host(sx).T, s_ref, f"dual kernel 1x128 scales (pow2={pow2})")


@pytest.mark.parametrize("transposed", [False, True])
@pytest.mark.parametrize("pow2", [False, True])
def test_weight_blocks_every_quotient(pow2, transposed):
    """One 128x128 block per absmax (every mantissa at eight exponents): the
    block holds _values_below(absmax) and the absmax; W[128, 128 * blocks]."""
    torch, fp8bs = require_gpu()
    blocks = []
    for e in (0, 20, 42, 43, 100, 127, 200, 254):
        for f in range(128):
            a = (e << 7) | f
            if a == 0:
                continue
            v = _values_below(a)
            blk = np.zeros(128 * 128, np.uint16)
            blk[0] = a | (np.uint16(0x8000) if f & 1 else np.uint16(0))
            blk[1: 1 + len(v)] = v
            rng = np.random.default_rng(a)
            blocks.append(rng.permutation(blk).reshape(128, 128))   # absmax anywhere in the block
    w_bits = np.ascontiguousarray(np.concatenate(blocks, axis=1))   # [128, 128 * nblocks]
    out = fp8bs.quantize_weight(to_dev_bf16(w_bits), transposed=transposed, pow2=pow2)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_get_device_status() == 0
    q_ref, s_ref = oracle.quantize_weight_128x128(w_bits, pow2=pow2)
    assert_bytes_equal(to_host(out[0]), q_ref, "weight codes")
    assert_scales_equal(to_host(out[1]), s_ref, "weight scales")
    if transposed:
        assert_bytes_equal(to_host(out[2]), np.ascontiguousarray(q_ref.T), "transposed weight codes")
        assert_scales_equal(to_host(out[3]), np.ascontiguousarray(s_ref.T), "transposed weight scales")
