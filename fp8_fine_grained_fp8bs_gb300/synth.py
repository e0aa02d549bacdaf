"""Seeded synthetic inputs shaped like the DeepSeek-V3 layers that the
fine-grained FP8 scheme is applied to.

This module is the only code shared by the CPU oracle side (tests, the
CPU baseline) and the CUDA side (tests, bench). It draws random numbers and
lays out workloads; it contains none of the quantisation or GEMM arithmetic.

Recipe (all seeded, deterministic for a given numpy version):
  * each tensor has its own stream: ``numpy.random.Generator(PCG64(SeedSequence([seed, tensor_id])))``;
  * normals: ``standard_normal`` in float32, times sigma;
  * outliers (activations only): every element independently with
    probability 1e-3 is multiplied by 50;
  * the float32 value is rounded to BF16 with round-to-nearest-even and kept
    as its uint16 bit pattern.

MoE routing (DeepSeek-V3 "Infrastructure" §3.3.3 low-precision
communication: activations are dispatched per expert before the up
projection): every token picks 8 distinct experts out of 32, drawn without
replacement with probability proportional to ``(e + 1) ** -1.1`` (a Zipf
law with s = 1.1).  Sequential weighted sampling without replacement is
drawn with the Gumbel-top-k construction, which has the same distribution.
Each expert's rows are contiguous and padded with zero rows to a multiple
of 128.
"""
from __future__ import annotations

import numpy as np

BF16 = np.uint16

# Tensor ids: one independent stream per tensor of a workload.
TID_X = 1
TID_W = 2
TID_X_LARGE = 3
TID_DY = 4
TID_W_GATE_UP = 5
TID_W_DOWN = 6
TID_ROUTING = 7
TID_DOWN_IN = 8
TID_GATE = 9
TID_OUTLIER = 1000  # added to the tensor id of the tensor that gets outliers

_CHUNK = 1 << 22


def _rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (nearest, ties to even); return uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(shape, sigma: float, seed: int, tensor_id: int, outliers: bool = False) -> np.ndarray:
    """BF16 bit patterns of sigma * N(0,1), optionally with 0.1% x50 outliers."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    g = _rng(seed, tensor_id)
    go = _rng(seed, tensor_id + TID_OUTLIER) if outliers else None
    sig = np.float32(sigma)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        v = g.standard_normal(hi - lo, dtype=np.float32) * sig
        if go is not None:
            hit = go.random(hi - lo, dtype=np.float32) < np.float32(1e-3)
            v[hit] *= np.float32(50.0)
        out[lo:hi] = f32_to_bf16_bits(v)
    return out.reshape(shape)


# ---------------------------------------------------------------- workloads

def tiny_fprop(seed: int = 0):
    """X[128,512] ~N(0,1) + outliers, W[256,512] ~N(0,0.02); FP32 out."""
    x = normal_bf16((128, 512), 1.0, seed, TID_X, outliers=True)
    w = normal_bf16((256, 512), 0.02, seed, TID_W)
    return x, w


def dense_fprop(seed: int = 0, M: int = 4096, N: int = 7168, K: int = 7168):
    """X[M,K] ~N(0,1) + outliers, W[N,K] ~N(0,0.02); BF16 out."""
    x = normal_bf16((M, K), 1.0, seed, TID_X, outliers=True)
    w = normal_bf16((N, K), 0.02, seed, TID_W)
    return x, w


def quantize_input(seed: int = 0, M: int = 16384, K: int = 7168):
    """The standalone activation-quantize input X[M,K] ~N(0,1) + outliers."""
    return normal_bf16((M, K), 1.0, seed, TID_X_LARGE, outliers=True)


def dgrad(seed: int = 0, M: int = 4096, K: int = 7168, N: int = 2048):
    """dY[M,K] ~N(0,1e-3) and W[K,N] ~N(0,0.02) (the Linear's weight, used transposed)."""
    dy = normal_bf16((M, K), 1e-3, seed, TID_DY)
    w = normal_bf16((K, N), 0.02, seed, TID_W)
    return dy, w


def wgrad(seed: int = 0, T: int = 16384, N: int = 2048, K: int = 7168):
    """dY[T,N] and X[T,K], both ~N(0,1)."""
    dy = normal_bf16((T, N), 1.0, seed, TID_DY)
    x = normal_bf16((T, K), 1.0, seed, TID_X)
    return dy, x


def moe_routing(seed: int = 0, tokens: int = 8192, experts: int = 32, top_k: int = 8,
                zipf_s: float = 1.1):
    """Expert choices [tokens, top_k] (distinct per token), Zipf-weighted."""
    g = _rng(seed, TID_ROUTING)
    logw = -zipf_s * np.log(np.arange(1, experts + 1, dtype=np.float64))
    gumbel = -np.log(-np.log(g.random((tokens, experts))))
    keys = logw[None, :] + gumbel
    return np.argsort(-keys, axis=1, kind="stable")[:, :top_k].astype(np.int32)


def moe_gate_weights(seed: int = 0, tokens: int = 8192, top_k: int = 8) -> np.ndarray:
    """Gate weights [tokens, top_k] float32 of the routed experts: positive,
    each token's weights normalised to sum to 1 (uniform draws in (0.05, 1))."""
    g = _rng(seed, TID_GATE)
    w = g.uniform(0.05, 1.0, (tokens, top_k)).astype(np.float32)
    return (w / w.sum(axis=1, keepdims=True)).astype(np.float32)


def moe_layout(choice: np.ndarray, experts: int = 32, align: int = 128):
    """Group the (token, expert) pairs by expert.

    Returns ``(offsets, src)``: ``offsets`` int32 [experts+1] row offsets of
    each expert's segment (multiples of ``align``); ``src`` int64 [rows]
    the source token of every row, -1 for a zero padding row.
    """
    tokens, top_k = choice.shape
    flat_e = choice.reshape(-1)
    flat_t = np.repeat(np.arange(tokens, dtype=np.int64), top_k)
    order = np.argsort(flat_e, kind="stable")
    counts = np.bincount(flat_e, minlength=experts)
    padded = (counts + align - 1) // align * align
    offsets = np.zeros(experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    src = np.full(int(offsets[-1]), -1, dtype=np.int64)
    start = 0
    for e in range(experts):
        c = int(counts[e])
        src[offsets[e]:offsets[e] + c] = flat_t[order[start:start + c]]
        start += c
    return offsets.astype(np.int32), src


def moe_fprop(seed: int = 0, tokens: int = 8192, experts: int = 32, top_k: int = 8,
              hidden: int = 7168, inter: int = 2048, with_weights: bool = True):
    """MoE grouped-GEMM workload.

    Returns a dict with ``x_tok`` [tokens, hidden] BF16 (token activations),
    ``offsets``/``src`` (the grouped row layout), ``w_gate_up`` [E, 2*inter, hidden],
    ``w_down`` [E, hidden, inter] and ``down_in`` [rows, inter] (synthetic
    down-projection input; zero on padding rows).
    """
    choice = moe_routing(seed, tokens, experts, top_k)
    offsets, src = moe_layout(choice, experts)
    out = {
        "x_tok": normal_bf16((tokens, hidden), 1.0, seed, TID_X, outliers=True),
        "offsets": offsets,
        "src": src,
    }
    if with_weights:
        out["w_gate_up"] = normal_bf16((experts, 2 * inter, hidden), 0.02, seed, TID_W_GATE_UP)
        out["w_down"] = normal_bf16((experts, hidden, inter), 0.02, seed, TID_W_DOWN)
        d = normal_bf16((int(offsets[-1]), inter), 1.0, seed, TID_DOWN_IN)
        d[src < 0] = 0
        out["down_in"] = d
    return out


def gather_rows(x_tok: np.ndarray, src: np.ndarray) -> np.ndarray:
    """Dispatch: row r of the result is token src[r], or zeros where src[r] < 0."""
    out = np.zeros((src.shape[0], x_tok.shape[1]), dtype=x_tok.dtype)
    ok = src >= 0
    out[ok] = x_tok[src[ok]]
    return out
