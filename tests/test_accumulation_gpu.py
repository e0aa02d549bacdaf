"""Accumulation precision without promotion, on the GPU.

DeepSeek-V3 §3.3.2 "Increasing accumulation precision" measures the FP8 GEMM
of the H800 tensor core with all of K accumulated inside the tensor core:
about 14 bits kept, a maximum relative error near 2% for K = 4096, which is
why the pages promote partial sums to FP32 every N_C = 128.  The diagnostic
entry fp8bs_diag_gemm_unpromoted runs that configuration on this GPU (all of
K accumulated in tensor memory); it is compared with the exact sum, which
float64 holds exactly here (every product of two E4M3 values is a multiple
of 2^-18 below 2^18, so 4096 of them need fewer than 53 bits), next to the
promoted production GEMM on the same codes.
"""
import numpy as np
import pytest

import oracle
from fp8_fine_grained_fp8bs_gb300 import synth
from _gpu import require_gpu, to_dev, to_host

pytestmark = pytest.mark.gpu


def _per_tensor_codes(shape, tensor_id):
    """N(0,1) BF16 values quantised with one scale for the whole tensor."""
    x = synth.normal_bf16(shape, 1.0, 31, tensor_id)
    codes, s = oracle.quantize_groups(x.reshape(1, -1))
    return codes.reshape(shape), float(s[0])


def _errors(got, Y):
    err = np.abs(np.asarray(got, np.float64) - Y)
    big = np.abs(Y) >= 0.1 * np.sqrt(np.mean(Y * Y))
    return float(err.max() / np.abs(Y).max()), float((err[big] / np.abs(Y[big])).max())


def test_unpromoted_k4096_is_fp32_grade():
    torch, fp8bs = require_gpu()
    M, N, K = 128, 256, 4096
    qa, _ = _per_tensor_codes((M, K), 1)
    qb, _ = _per_tensor_codes((N, K), 2)
    A, B = oracle.e4m3_decode(qa), oracle.e4m3_decode(qb)
    Y = A @ B.T                                   # exact (see the module docstring)
    T = np.abs(A) @ np.abs(B).T
    d_unprom = to_host(fp8bs.diag_gemm_unpromoted(to_dev(qa), to_dev(qb)))
    assert fp8bs.fp8bs_get_device_status() == 0
    # the promoted production GEMM on the same codes: every block scale 1
    ones_a = to_dev(np.ones((K // 128, M), np.float32))
    ones_b = to_dev(np.ones((N // 128, K // 128), np.float32))
    d_prom = to_host(fp8bs.gemm(to_dev(qa), ones_a, to_dev(qb), ones_b, out_dtype=torch.float32))
    e_un, r_un = _errors(d_unprom, Y)
    e_pr, r_pr = _errors(d_prom, Y)
    print(f"\nK=4096 no promotion: max|err|/max|Y| {e_un:.2e}, max rel err {r_un:.2e}; "
          f"promoted every 128 K: {e_pr:.2e}, {r_pr:.2e}; pages (H800, no promotion): about 2e-2")
    # FP32-grade without promotion, three orders of magnitude below the pages' H800 figure
    assert e_un < 1e-5 and r_un < 1e-4
    assert np.all(np.abs(d_prom - Y) <= 1e-5 * T)


def test_unpromoted_tiles_every_element():
    """Several 128x256 tiles in both directions, short K: every element within
    FP32 accumulation error of the exact sum."""
    torch, fp8bs = require_gpu()
    M, N, K = 384, 512, 384
    qa, _ = _per_tensor_codes((M, K), 3)
    qb, _ = _per_tensor_codes((N, K), 4)
    A, B = oracle.e4m3_decode(qa), oracle.e4m3_decode(qb)
    Y = A @ B.T
    T = np.abs(A) @ np.abs(B).T
    d = to_host(fp8bs.diag_gemm_unpromoted(to_dev(qa), to_dev(qb)))
    assert fp8bs.fp8bs_get_device_status() == 0
    assert np.all(np.abs(d - Y) <= 1e-5 * T)
