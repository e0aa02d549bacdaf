"""Online absmax quantisation to E4M3, per group.

TEST INFRASTRUCTURE ONLY (see the package docstring).

DeepSeek-V3 §3.3.2 "fine-grained quantization" and "online quantization":
the max absolute value of every group is computed at use time, the scale
is derived from it and the values are cast to FP8.  Groups:
  * activations: 1 x 128 (one token, 128 consecutive channels);
  * weights: 128 x 128 (128 output channels x 128 input channels);
  * the backward pass also needs activations grouped 128 x 1 (128
    consecutive tokens of one channel) — §3.3.3 "low-precision activations"
    (1) and §3.5.2 "support for transposed GEMM operations".
Formulas from the Figure 7 explainer ("Fine-grained quantization"):
s = absmax(group) / F_max and FP8(x) = round(x / s), with F_max = 448.

Power-of-two ("rounded") scales: §3.3.3 "low-precision activations" (1)
and "low-precision communication" use scaling factors that are integer
powers of two for activations that are later re-tiled from 1x128 to 128x1
(and for the activations dispatched before the MoE up-projection), so the
re-tiling adds no quantisation error.  Read here as the smallest power of
two s = 2^k with absmax / s <= 448 (no value saturates), k clamped to the
float32 range (k >= -149); codes are E4M3(fl32(x / s)) as before.

Re-tiling (§3.5.2 "support for transposed GEMM operations"): the backward
pass reads the 1x128-quantised activations, dequantises them, transposes
and requantises them in 128x1 groups.  The dequantised value is
fl32(dec(code) * s) (exact for power-of-two scales).

Layouts returned here are the logical ones:
  quantize_act_1x128(X[M,K])   -> codes [M,K], scales [M, K/128]
  quantize_act_128x1(X[M,K])   -> codes of X^T [K,M], scales [K, M/128]
  quantize_weight_128x128(W[N,K]) -> codes [N,K], scales [N/128, K/128]
  requant_1x128_to_128x1(codes [M,K], scales [M,K/128]) -> codes of X^T [K,M], scales [K, M/128]
"""
from __future__ import annotations

import numpy as np

from .e4m3 import E4M3_MAX, e4m3_decode, e4m3_encode

GROUP = 128


def bf16_bits_to_f32(b) -> np.ndarray:
    """BF16 bit patterns (uint16) widened to float32; exact."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _as_f32(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_bits_to_f32(x)
    if x.dtype != np.float32:
        raise TypeError("inputs are BF16 bit patterns (uint16) or float32")
    return x


MIN_POW2_EXP = -149   # 2^-149: the smallest positive float32


def pow2_scale(a) -> np.ndarray:
    """Smallest power of two 2^k with a / 2^k <= 448 (k >= -149), as float32; 0 where a == 0.

    The candidate exponent from a floating-point log is corrected with exact
    comparisons (448 * 2^k and a are both exact in float64).
    """
    a = np.asarray(a, dtype=np.float64)
    pos = a > 0
    safe = np.where(pos, a, 1.0)
    k = np.ceil(np.log2(safe / E4M3_MAX)).astype(np.int64)
    for _ in range(2):
        k = np.where(np.ldexp(E4M3_MAX, k - 1) >= safe, k - 1, k)   # a smaller power still suffices
        k = np.where(np.ldexp(E4M3_MAX, k) < safe, k + 1, k)        # not yet large enough
    k = np.maximum(k, MIN_POW2_EXP)
    return np.where(pos, np.ldexp(1.0, k), 0.0).astype(np.float32)   # exact: 2^k >= 2^-149


def quantize_groups(g, pow2: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """Quantise each row of ``g`` [G, n] as one group.

    absmax is exact; s = fl32(absmax / 448) (IEEE float32 division), or with
    ``pow2`` the power-of-two scale of ``pow2_scale``; code = E4M3(fl32(x / s));
    a group with s == 0 gets all-zero codes.
    """
    g = _as_f32(g)
    a = np.max(np.abs(g), axis=1)                                # exact
    if pow2:
        s = pow2_scale(a)
    else:
        s = (a / np.float32(E4M3_MAX)).astype(np.float32)        # float32 / float32, IEEE RN
    with np.errstate(divide="ignore", invalid="ignore"):
        y = (g / s[:, None]).astype(np.float32)                  # float32 / float32, IEEE RN
    codes = e4m3_encode(np.where(s[:, None] > 0, y, np.float32(0.0)))
    codes[s == 0] = 0
    return codes, s


def quantize_act_1x128(x, pow2: bool = False):
    """1x128 tiles along the rows of X[M,K] (K % 128 == 0)."""
    x = _as_f32(x)
    M, K = x.shape
    assert K % GROUP == 0
    codes, s = quantize_groups(x.reshape(M * (K // GROUP), GROUP), pow2)
    return codes.reshape(M, K), s.reshape(M, K // GROUP)


def quantize_act_128x1(x, pow2: bool = False):
    """128x1 tiles: 128 consecutive rows of one column of X[M,K] (M % 128 == 0).

    Returns the codes of X^T, [K, M], and scales [K, M/128]: the result is
    the 1x128 quantisation of X^T.
    """
    x = _as_f32(x)
    M, K = x.shape
    assert M % GROUP == 0
    return quantize_act_1x128(np.ascontiguousarray(x.T), pow2)


def dequantize_1x128(codes, scales) -> np.ndarray:
    """fl32(dec(code) * s) of 1x128-quantised X: codes [M,K], scales [M,K/128] -> float32 [M,K]."""
    dec = e4m3_decode(codes).astype(np.float32)                 # exact: every E4M3 value is a float32
    s = np.repeat(np.asarray(scales, dtype=np.float32), GROUP, axis=1)
    return (dec * s).astype(np.float32)                          # float32 * float32, IEEE RN


def requant_1x128_to_128x1(codes, scales, pow2: bool = True):
    """Backward re-tiling: dequantise 1x128-quantised X[M,K], transpose, and
    requantise in 128x1 groups (M % 128 == 0).  Returns the codes of X^T
    [K, M] and scales [K, M/128], like ``quantize_act_128x1``."""
    return quantize_act_128x1(dequantize_1x128(codes, scales), pow2)


def quantize_weight_128x128(w, pow2: bool = False):
    """128x128 blocks of W[N,K] (N % 128 == 0, K % 128 == 0)."""
    w = _as_f32(w)
    N, K = w.shape
    assert N % GROUP == 0 and K % GROUP == 0
    nb, kb = N // GROUP, K // GROUP
    blocks = w.reshape(nb, GROUP, kb, GROUP).transpose(0, 2, 1, 3).reshape(nb * kb, GROUP * GROUP)
    codes, s = quantize_groups(blocks, pow2)
    codes = codes.reshape(nb, kb, GROUP, GROUP).transpose(0, 2, 1, 3).reshape(N, K)
    return codes, s.reshape(nb, kb)


def swiglu(h, inter: int) -> np.ndarray:
    """SwiGLU of the MoE gate/up projection output, in float64.

    DeepSeek-V3 §3.3.3 "low-precision activations" (2): the input of the
    MoE SwiGLU operator is cached and its output recomputed; the output
    feeds the down projection, whose input is quantised 1x128.  ``h`` is
    [M, 2*inter] (BF16 bits or float32) with the gate projection in columns
    [0, inter) and the up projection in [inter, 2*inter):
        out = silu(gate) * up,   silu(g) = g / (1 + exp(-g)).
    """
    h = _as_f32(h).astype(np.float64)
    g, u = h[:, :inter], h[:, inter:2 * inter]
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


def bf16_round_f64(v) -> np.ndarray:
    """Nearest BF16 value (ties to even) of float64 values, as float32; exact."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(ex.astype(np.int64) - 1, -126)    # BF16 shares float32's exponent range
    quantum = np.exp2((e - 7).astype(np.float64))
    r = np.rint(a / quantum) * quantum               # a / quantum is exact; rint: ties to even
    return np.copysign(r, v).astype(np.float32)      # exact: r has <= 8 significant bits


def swiglu_quantize_1x128(h, inter: int, pow2: bool = False):
    """The 1x128 quantisation of the BF16-rounded SwiGLU output (the unfused
    pipeline: SwiGLU -> BF16 activation -> 1x128 quantise)."""
    return quantize_act_1x128(bf16_round_f64(swiglu(h, inter)), pow2)
