"""Python binding of the fp8bs C ABI (include/fp8bs.h).

Fine-grained FP8 quantisation and block-scaled FP8 GEMM on GB300 (sm_103a),
after DeepSeek-V3 "Infrastructure" §3.3.  Every step runs in the CUDA
library ``_build/libfp8bs.so``; this module only marshals arguments
(tensors -> device pointers, the current torch stream) and turns non-zero
status codes into exceptions.  There is no CPU path: if the library is
missing or fails to load, every call raises.

The functions named ``fp8bs_*`` mirror the C entry points one to one and
take tensors or raw device pointers.  ``quantize_act``, ``quantize_weight``,
``gemm`` and ``grouped_gemm`` additionally allocate their outputs with torch.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH, build as _build

__all__ = [
    "Fp8bsError", "load_library", "build",
    "fp8bs_quantize_act", "fp8bs_quantize_weight", "fp8bs_gemm", "fp8bs_grouped_gemm",
    "fp8bs_gemm_pow2", "fp8bs_grouped_gemm_pow2",
    "fp8bs_gather_q_rows", "fp8bs_scatter_q_rows", "fp8bs_gather_bf16_rows", "fp8bs_moe_combine", "SCALES_KB_MAJOR",
    "SCALES_ROW_MAJOR",
    "fp8bs_quantize_act_ex", "fp8bs_quantize_weight_ex", "fp8bs_quantize_act_weight", "quantize_act_weight", "fp8bs_requant_1x128_to_128x1", "fp8bs_swiglu_quantize",
    "fp8bs_get_device_status", "fp8bs_set_wait_timeout_ms", "fp8bs_status_string", "fp8bs_selftest_wait_timeout",
    "fp8bs_diag_gemm_unpromoted", "diag_gemm_unpromoted",
    "quantize_act", "quantize_weight", "gemm", "grouped_gemm", "requant_1x128_to_128x1", "swiglu_quantize",
    "OUT_F32", "OUT_BF16", "SCALE_BLOCK128x128", "SCALE_ROW1x128", "SCALE_ABSMAX", "SCALE_POW2",
]

OUT_F32, OUT_BF16 = 0, 1
SCALES_KB_MAJOR, SCALES_ROW_MAJOR = 0, 1
SCALE_BLOCK128x128, SCALE_ROW1x128 = 0, 1
SCALE_ABSMAX, SCALE_POW2 = 0, 1

STATUS_NAMES = {0: "FP8BS_OK", 1: "FP8BS_ERR_INVALID_ARG", 2: "FP8BS_ERR_SHAPE", 3: "FP8BS_ERR_ALIGNMENT",
                4: "FP8BS_ERR_UNSUPPORTED_ARCH", 5: "FP8BS_ERR_CUDA", 6: "FP8BS_ERR_TIMEOUT",
                7: "FP8BS_ERR_DEVICE_ARG"}


class Fp8bsError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


_lib = None
_lock = threading.Lock()

_c_i64, _c_int, _c_vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
_SIGNATURES = {
    "fp8bs_quantize_act": [_c_vp, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp],
    "fp8bs_quantize_weight": [_c_vp, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp],
    "fp8bs_quantize_act_ex": [_c_vp, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_vp],
    "fp8bs_quantize_weight_ex": [_c_vp, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_vp],
    "fp8bs_quantize_act_weight": [_c_vp, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64,
                                  _c_vp, _c_vp, _c_int, _c_vp],
    "fp8bs_requant_1x128_to_128x1": [_c_vp, _c_vp, _c_i64, _c_i64, _c_vp, _c_vp, _c_int, _c_vp],
    "fp8bs_swiglu_quantize": [_c_vp, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp, _c_int, _c_vp],
    "fp8bs_gemm": [_c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_vp, _c_int, _c_i64, _c_i64, _c_i64, _c_int, _c_vp],
    "fp8bs_grouped_gemm": [_c_vp, _c_vp, _c_i64, _c_vp, _c_int, _c_vp, _c_vp, _c_vp, _c_int, _c_i64, _c_i64,
                           _c_vp],
    "fp8bs_gemm_pow2": [_c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_vp, _c_int, _c_i64, _c_i64, _c_i64, _c_int, _c_vp],
    "fp8bs_grouped_gemm_pow2": [_c_vp, _c_vp, _c_i64, _c_vp, _c_int, _c_vp, _c_vp, _c_vp, _c_int, _c_i64, _c_i64,
                                _c_vp],
    "fp8bs_gather_q_rows": [_c_vp, _c_vp, _c_i64, _c_i64, _c_int, _c_vp, _c_i64, _c_vp, _c_vp, _c_int, _c_vp],
    "fp8bs_scatter_q_rows": [_c_vp, _c_vp, _c_i64, _c_i64, _c_int, _c_vp, _c_int, _c_vp, _c_i64, _c_i64, _c_vp, _c_vp,
                             _c_int, _c_vp],
    "fp8bs_gather_bf16_rows": [_c_vp, _c_i64, _c_i64, _c_vp, _c_i64, _c_vp, _c_vp],
    "fp8bs_moe_combine": [_c_vp, _c_i64, _c_i64, _c_vp, _c_vp, _c_i64, _c_int, _c_vp, _c_vp],
    "fp8bs_get_device_status": [_c_vp],
    "fp8bs_selftest_wait_timeout": [_c_i64, _c_vp],
    "fp8bs_diag_gemm_unpromoted": [_c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_vp],
    "fp8bs_set_wait_timeout_ms": [_c_i64],
    "fp8bs_status_string": [_c_int],
}


def build(force: bool = False) -> str:
    """Compiles the CUDA library in-tree (nvcc, sm_103a) and returns its path."""
    return _build(force=force)


def load_library(path: str | None = None):
    """Loads libfp8bs.so (raises if it is missing: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"fp8bs CUDA library not built: {p} is missing (run build())")
            lib = ctypes.CDLL(p, mode=ctypes.RTLD_LOCAL)
            for name, argtypes in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = argtypes
                fn.restype = ctypes.c_char_p if name == "fp8bs_status_string" else ctypes.c_int
            _lib = lib
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != 0:
        raise Fp8bsError(status, where)


# ------------------------------------------------------------ raw C entry points

def fp8bs_quantize_act(x, M, K, ldx, xq, sx, xq_t=None, sx_t=None, stream=None):
    lib = load_library()
    _check(lib.fp8bs_quantize_act(_ptr(x), M, K, ldx, _ptr(xq), _ptr(sx), _ptr(xq_t), _ptr(sx_t),
                                  _stream(stream)), "fp8bs_quantize_act")


def fp8bs_quantize_weight(w, N, K, ldw, wq, sw, wq_t=None, sw_t=None, stream=None):
    lib = load_library()
    _check(lib.fp8bs_quantize_weight(_ptr(w), N, K, ldw, _ptr(wq), _ptr(sw), _ptr(wq_t), _ptr(sw_t),
                                     _stream(stream)), "fp8bs_quantize_weight")


def fp8bs_quantize_act_ex(x, M, K, ldx, xq, sx, xq_t=None, sx_t=None, scale_mode=SCALE_ABSMAX, stream=None):
    lib = load_library()
    _check(lib.fp8bs_quantize_act_ex(_ptr(x), M, K, ldx, _ptr(xq), _ptr(sx), _ptr(xq_t), _ptr(sx_t),
                                     int(scale_mode), _stream(stream)), "fp8bs_quantize_act_ex")


def fp8bs_quantize_weight_ex(w, N, K, ldw, wq, sw, wq_t=None, sw_t=None, scale_mode=SCALE_ABSMAX, stream=None):
    lib = load_library()
    _check(lib.fp8bs_quantize_weight_ex(_ptr(w), N, K, ldw, _ptr(wq), _ptr(sw), _ptr(wq_t), _ptr(sw_t),
                                        int(scale_mode), _stream(stream)), "fp8bs_quantize_weight_ex")


def fp8bs_requant_1x128_to_128x1(xq, sx, M, K, xq_t, sx_t, scale_mode=SCALE_POW2, stream=None):
    lib = load_library()
    _check(lib.fp8bs_requant_1x128_to_128x1(_ptr(xq), _ptr(sx), M, K, _ptr(xq_t), _ptr(sx_t), int(scale_mode),
                                            _stream(stream)), "fp8bs_requant_1x128_to_128x1")


def fp8bs_swiglu_quantize(h, M, I, ldh, q, s, scale_mode=SCALE_ABSMAX, stream=None):
    lib = load_library()
    _check(lib.fp8bs_swiglu_quantize(_ptr(h), M, I, ldh, _ptr(q), _ptr(s), int(scale_mode), _stream(stream)),
           "fp8bs_swiglu_quantize")


def fp8bs_gemm(a, sa, b, sb, sb_kind, d, d_dtype, M, N, K, accumulate=0, stream=None):
    lib = load_library()
    _check(lib.fp8bs_gemm(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), sb_kind, _ptr(d), d_dtype, M, N, K,
                          int(accumulate), _stream(stream)), "fp8bs_gemm")


def fp8bs_grouped_gemm(a, sa, M_total, offsets, num_groups, b, sb, d, d_dtype, N, K, stream=None):
    lib = load_library()
    _check(lib.fp8bs_grouped_gemm(_ptr(a), _ptr(sa), M_total, _ptr(offsets), num_groups, _ptr(b), _ptr(sb),
                                  _ptr(d), d_dtype, N, K, _stream(stream)), "fp8bs_grouped_gemm")


def fp8bs_gemm_pow2(a, sa, b, sb, sb_kind, d, d_dtype, M, N, K, accumulate=0, stream=None):
    lib = load_library()
    _check(lib.fp8bs_gemm_pow2(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), sb_kind, _ptr(d), d_dtype, M, N, K,
                               int(accumulate), _stream(stream)), "fp8bs_gemm_pow2")


def fp8bs_grouped_gemm_pow2(a, sa, M_total, offsets, num_groups, b, sb, d, d_dtype, N, K, stream=None):
    lib = load_library()
    _check(lib.fp8bs_grouped_gemm_pow2(_ptr(a), _ptr(sa), M_total, _ptr(offsets), num_groups, _ptr(b), _ptr(sb),
                                       _ptr(d), d_dtype, N, K, _stream(stream)), "fp8bs_grouped_gemm_pow2")


def fp8bs_gather_q_rows(q, s, rows_in, H, s_in_layout, idx, rows_out, q_out, s_out, s_out_layout, stream=None):
    _check(load_library().fp8bs_gather_q_rows(_ptr(q), _ptr(s), rows_in, H, int(s_in_layout), _ptr(idx), rows_out,
                                              _ptr(q_out), _ptr(s_out), int(s_out_layout), _stream(stream)),
           "fp8bs_gather_q_rows")


def fp8bs_scatter_q_rows(q, s, rows_in, H, s_in_layout, pos, k, zero_rows, n_zero, rows_out, q_out, s_out,
                         s_out_layout, stream=None):
    _check(load_library().fp8bs_scatter_q_rows(_ptr(q), _ptr(s), rows_in, H, int(s_in_layout), _ptr(pos), int(k),
                                               _ptr(zero_rows), n_zero, rows_out, _ptr(q_out), _ptr(s_out),
                                               int(s_out_layout), _stream(stream)),
           "fp8bs_scatter_q_rows")


def fp8bs_gather_bf16_rows(y, rows_in, N, idx, rows_out, out, stream=None):
    _check(load_library().fp8bs_gather_bf16_rows(_ptr(y), rows_in, N, _ptr(idx), rows_out, _ptr(out), _stream(stream)),
           "fp8bs_gather_bf16_rows")


def fp8bs_moe_combine(y, rows_y, N, idx, w, T, k, out, stream=None):
    _check(load_library().fp8bs_moe_combine(_ptr(y), rows_y, N, _ptr(idx), _ptr(w), T, int(k), _ptr(out),
                                            _stream(stream)), "fp8bs_moe_combine")


def fp8bs_get_device_status(stream=None) -> int:
    return load_library().fp8bs_get_device_status(_stream(stream))


def fp8bs_selftest_wait_timeout(timeout_us: int, stream=None):
    _check(load_library().fp8bs_selftest_wait_timeout(int(timeout_us), _stream(stream)), "fp8bs_selftest_wait_timeout")


def fp8bs_quantize_act_weight(x, M, K, ldx, xq, sx, w, N, Kw, ldw, wq, sw, scale_mode=0, stream=None):
    _check(load_library().fp8bs_quantize_act_weight(_ptr(x), M, K, ldx, _ptr(xq), _ptr(sx), _ptr(w), N, Kw, ldw,
                                                    _ptr(wq), _ptr(sw), int(scale_mode), _stream(stream)),
           "fp8bs_quantize_act_weight")


def fp8bs_diag_gemm_unpromoted(a, b, d, M, N, K, stream=None):
    _check(load_library().fp8bs_diag_gemm_unpromoted(_ptr(a), _ptr(b), _ptr(d), M, N, K, _stream(stream)),
           "fp8bs_diag_gemm_unpromoted")


def fp8bs_set_wait_timeout_ms(ms: int):
    _check(load_library().fp8bs_set_wait_timeout_ms(int(ms)), "fp8bs_set_wait_timeout_ms")


def fp8bs_status_string(status: int) -> str:
    return load_library().fp8bs_status_string(int(status)).decode()


# ------------------------------------------------------ allocating conveniences

def quantize_act(x, transposed: bool = False, pow2: bool = False, stream=None):
    """x: [M, K] bfloat16 CUDA tensor (row-major, K % 128 == 0).

    Returns (xq [M,K] uint8, sx [K/128, M] float32) and, with ``transposed``,
    also (xq_t [K,M] uint8, sx_t [M/128, K] float32).  ``pow2`` selects
    power-of-two scales (SCALE_POW2).
    """
    import torch
    M, K = x.shape
    xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    sx = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    xq_t = sx_t = None
    if transposed:
        xq_t = torch.empty((K, M), dtype=torch.uint8, device=x.device)
        sx_t = torch.empty((M // 128, K), dtype=torch.float32, device=x.device)
    fp8bs_quantize_act_ex(x, M, K, x.stride(0), xq, sx, xq_t, sx_t, SCALE_POW2 if pow2 else SCALE_ABSMAX, stream)
    return (xq, sx, xq_t, sx_t) if transposed else (xq, sx)


def quantize_weight(w, transposed: bool = False, pow2: bool = False, stream=None):
    """w: [N, K] bfloat16 CUDA tensor.  Returns (wq, sw[, wq_t, sw_t])."""
    import torch
    N, K = w.shape
    wq = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)
    wq_t = sw_t = None
    if transposed:
        wq_t = torch.empty((K, N), dtype=torch.uint8, device=w.device)
        sw_t = torch.empty((K // 128, N // 128), dtype=torch.float32, device=w.device)
    fp8bs_quantize_weight_ex(w, N, K, w.stride(0), wq, sw, wq_t, sw_t, SCALE_POW2 if pow2 else SCALE_ABSMAX, stream)
    return (wq, sw, wq_t, sw_t) if transposed else (wq, sw)


def swiglu_quantize(h, pow2: bool = False, stream=None):
    """h: [M, 2I] bfloat16 CUDA tensor (gate | up).  Returns (q [M, I] uint8,
    s [I/128, M] float32): the 1x128 quantisation of BF16(silu(gate) * up)."""
    import torch
    M, two_i = h.shape
    I = two_i // 2
    q = torch.empty((M, I), dtype=torch.uint8, device=h.device)
    s = torch.empty((I // 128, M), dtype=torch.float32, device=h.device)
    fp8bs_swiglu_quantize(h, M, I, h.stride(0), q, s, SCALE_POW2 if pow2 else SCALE_ABSMAX, stream)
    return q, s


def requant_1x128_to_128x1(xq, sx, pow2: bool = True, stream=None):
    """Re-tile 1x128-quantised activations (xq [M,K] uint8, sx [K/128, M]) into
    128x1 groups: returns (xq_t [K,M] uint8, sx_t [M/128, K] float32)."""
    import torch
    M, K = xq.shape
    xq_t = torch.empty((K, M), dtype=torch.uint8, device=xq.device)
    sx_t = torch.empty((M // 128, K), dtype=torch.float32, device=xq.device)
    fp8bs_requant_1x128_to_128x1(xq, sx, M, K, xq_t, sx_t, SCALE_POW2 if pow2 else SCALE_ABSMAX, stream)
    return xq_t, sx_t


def gemm(a, sa, b, sb, sb_kind: int = SCALE_BLOCK128x128, out_dtype=None, out=None, accumulate: bool = False,
         stream=None, pow2: bool = False):
    """D = A B^T with per-128-K-block scales; A [M,K], B [N,K] uint8 E4M3.
    ``pow2``: power-of-two scales applied by the tensor core (fp8bs_gemm_pow2)."""
    import torch
    M, K = a.shape
    N = b.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, device=a.device)
    d_dtype = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    fn = fp8bs_gemm_pow2 if pow2 else fp8bs_gemm
    fn(a, sa, b, sb, sb_kind, out, d_dtype, M, N, K, int(accumulate), stream)
    return out


def grouped_gemm(a, sa, offsets, b, sb, out_dtype=None, out=None, stream=None, pow2: bool = False):
    """Per-expert D rows = A rows of the expert x B[g]^T; offsets: int32 CUDA tensor [G+1].
    ``pow2``: power-of-two scales applied by the tensor core (fp8bs_grouped_gemm_pow2)."""
    import torch
    M, K = a.shape
    G, N, _ = b.shape
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, device=a.device)
    d_dtype = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    fn = fp8bs_grouped_gemm_pow2 if pow2 else fp8bs_grouped_gemm
    fn(a, sa, M, offsets, G, b, sb, out, d_dtype, N, K, stream)
    return out


def diag_gemm_unpromoted(a, b, stream=None):
    """Diagnostic: FP32 D = A B^T of E4M3 codes (A [M,K], B [N,K] uint8) with all
    of K accumulated by the tensor core alone, no promotion and no scales."""
    import torch
    M, K = a.shape
    N = b.shape[0]
    out = torch.empty((M, N), dtype=torch.float32, device=a.device)
    fp8bs_diag_gemm_unpromoted(a, b, out, M, N, K, stream)
    return out


def quantize_act_weight(x, w, pow2: bool = False, stream=None):
    """X [M,K] and W [N,Kw] bfloat16 CUDA tensors quantised in one launch:
    returns (xq, sx [K/128, M], wq, sw [N/128, Kw/128])."""
    import torch
    M, K = x.shape
    N, Kw = w.shape
    xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    sx = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    wq = torch.empty((N, Kw), dtype=torch.uint8, device=w.device)
    sw = torch.empty((N // 128, Kw // 128), dtype=torch.float32, device=w.device)
    fp8bs_quantize_act_weight(x, M, K, x.stride(0), xq, sx, w, N, Kw, w.stride(0), wq, sw,
                              SCALE_POW2 if pow2 else SCALE_ABSMAX, stream)
    return xq, sx, wq, sw
