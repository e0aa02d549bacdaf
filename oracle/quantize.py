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

Layouts returned here are the logical ones:
  quantize_act_1x128(X[M,K])   -> codes [M,K], scales [M, K/128]
  quantize_act_128x1(X[M,K])   -> codes of X^T [K,M], scales [K, M/128]
  quantize_weight_128x128(W[N,K]) -> codes [N,K], scales [N/128, K/128]
"""
from __future__ import annotations

import numpy as np

from .e4m3 import E4M3_MAX, e4m3_encode

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


def quantize_groups(g) -> tuple[np.ndarray, np.ndarray]:
    """Quantise each row of ``g`` [G, n] as one group.

    absmax is exact; s = fl32(absmax / 448) (IEEE float32 division);
    code = E4M3(fl32(x / s)); a group with s == 0 gets all-zero codes.
    """
    g = _as_f32(g)
    a = np.max(np.abs(g), axis=1)                                # exact
    s = (a / np.float32(E4M3_MAX)).astype(np.float32)            # float32 / float32, IEEE RN
    with np.errstate(divide="ignore", invalid="ignore"):
        y = (g / s[:, None]).astype(np.float32)                  # float32 / float32, IEEE RN
    codes = e4m3_encode(np.where(s[:, None] > 0, y, np.float32(0.0)))
    codes[s == 0] = 0
    return codes, s


def quantize_act_1x128(x):
    """1x128 tiles along the rows of X[M,K] (K % 128 == 0)."""
    x = _as_f32(x)
    M, K = x.shape
    assert K % GROUP == 0
    codes, s = quantize_groups(x.reshape(M * (K // GROUP), GROUP))
    return codes.reshape(M, K), s.reshape(M, K // GROUP)


def quantize_act_128x1(x):
    """128x1 tiles: 128 consecutive rows of one column of X[M,K] (M % 128 == 0).

    Returns the codes of X^T, [K, M], and scales [K, M/128]: the result is
    the 1x128 quantisation of X^T.
    """
    x = _as_f32(x)
    M, K = x.shape
    assert M % GROUP == 0
    return quantize_act_1x128(np.ascontiguousarray(x.T))


def quantize_weight_128x128(w):
    """128x128 blocks of W[N,K] (N % 128 == 0, K % 128 == 0)."""
    w = _as_f32(w)
    N, K = w.shape
    assert N % GROUP == 0 and K % GROUP == 0
    nb, kb = N // GROUP, K // GROUP
    blocks = w.reshape(nb, GROUP, kb, GROUP).transpose(0, 2, 1, 3).reshape(nb * kb, GROUP * GROUP)
    codes, s = quantize_groups(blocks)
    codes = codes.reshape(nb, kb, GROUP, GROUP).transpose(0, 2, 1, 3).reshape(N, K)
    return codes, s.reshape(nb, kb)
