"""The C-ABI library builds, loads, exports every entry point declared in
include/fp8bs.h, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

import fp8_fine_grained_fp8bs_gb300 as fp8bs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fname in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fname.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fname)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(fp8bs_[a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    fp8bs.build()
    return fp8bs.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"fp8bs_quantize_act", "fp8bs_quantize_weight", "fp8bs_gemm", "fp8bs_grouped_gemm"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_only_the_abi_is_exported(lib):
    out = os.popen(f"nm -D --defined-only {fp8bs.build()}").read()
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert exported == set(_declared_functions())


def test_status_strings(lib):
    for s in range(8):
        assert fp8bs.fp8bs_status_string(s) not in ("", "unknown status")
    assert fp8bs.fp8bs_status_string(99) == "unknown status"


FAKE = 1 << 20          # 16-byte aligned, never dereferenced: every call below fails its checks first


@pytest.mark.parametrize("args,status", [
    ((FAKE, -1, 128, 128, FAKE, FAKE, None, None, None), 1),
    ((FAKE, 128, 100, 128, FAKE, FAKE, None, None, None), 2),
    ((FAKE, 100, 128, 128, FAKE, FAKE, FAKE, FAKE, None), 2),      # 128x1 needs M % 128 == 0
    ((FAKE, 128, 128, 128, FAKE, FAKE, FAKE, None, None), 1),      # xq_t without sx_t
    ((FAKE + 2, 128, 128, 128, FAKE, FAKE, None, None, None), 3),
    ((FAKE, 128, 128, 132, FAKE, FAKE, None, None, None), 3),      # ldx * 2 not a multiple of 16
    ((FAKE, 128, 256, 128, FAKE, FAKE, None, None, None), 1),      # ldx < K
    ((None, 128, 128, 128, FAKE, FAKE, None, None, None), 1),
])
def test_quantize_act_argument_errors(lib, args, status):
    assert lib.fp8bs_quantize_act(*args) == status


def test_quantize_weight_argument_errors(lib):
    assert lib.fp8bs_quantize_weight(FAKE, 100, 128, 128, FAKE, FAKE, None, None, None) == 2
    assert lib.fp8bs_quantize_weight(FAKE, 128, 128, 128, FAKE, FAKE, FAKE, None, None) == 1
    assert lib.fp8bs_quantize_weight(FAKE, 128, 128, 128, FAKE + 8, FAKE, None, None, None) == 3


def test_scale_mode_and_requant_argument_errors(lib):
    qa, qw, rq = lib.fp8bs_quantize_act_ex, lib.fp8bs_quantize_weight_ex, lib.fp8bs_requant_1x128_to_128x1
    assert qa(FAKE, 128, 128, 128, FAKE, FAKE, None, None, 2, None) == 1          # unknown scale mode
    assert qa(FAKE, 128, 100, 128, FAKE, FAKE, None, None, 1, None) == 2
    assert qw(FAKE, 128, 128, 128, FAKE, FAKE, None, None, -1, None) == 1
    assert qw(FAKE, 100, 128, 128, FAKE, FAKE, None, None, 1, None) == 2
    assert rq(FAKE, FAKE, 100, 128, FAKE, FAKE, 1, None) == 2                     # M % 128
    assert rq(FAKE, FAKE, 128, 100, FAKE, FAKE, 1, None) == 2                     # K % 128
    assert rq(FAKE, FAKE, 128, 128, FAKE, FAKE, 3, None) == 1                     # scale mode
    assert rq(FAKE, None, 128, 128, FAKE, FAKE, 1, None) == 1
    assert rq(FAKE, FAKE, 128, 128, FAKE + 8, FAKE, 1, None) == 3
    assert rq(FAKE, FAKE, -128, 128, FAKE, FAKE, 1, None) == 1
    assert rq(None, None, 0, 128, None, None, 1, None) == 0                       # empty: no-op


def test_swiglu_quantize_argument_errors(lib):
    sq = lib.fp8bs_swiglu_quantize
    assert sq(FAKE, 128, 256, 384, FAKE, FAKE, 0, None) == 1                      # ldh < 2I
    assert sq(FAKE, 128, 192, 384, FAKE, FAKE, 0, None) == 2                      # I % 128
    assert sq(FAKE, 128, 128, 256, FAKE, FAKE, 7, None) == 1                      # scale mode
    assert sq(FAKE, 128, 128, 260, FAKE, FAKE, 0, None) == 3                      # ldh * 2 % 16
    assert sq(FAKE + 4, 128, 128, 256, FAKE, FAKE, 0, None) == 3
    assert sq(None, 128, 128, 256, FAKE, FAKE, 0, None) == 1
    assert sq(None, 0, 128, 256, None, None, 0, None) == 0                        # empty: no-op


@pytest.mark.parametrize("name", ["fp8bs_gemm", "fp8bs_gemm_pow2"])
def test_gemm_argument_errors(lib, name):
    g = getattr(lib, name)
    assert g(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 0, 128, 128, 100, 0, None) == 2   # K % 128
    assert g(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 0, 128, 100, 128, 0, None) == 2   # N % 128
    assert g(FAKE, FAKE, FAKE, FAKE, 2, FAKE, 0, 128, 128, 128, 0, None) == 1   # scale kind
    assert g(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 5, 128, 128, 128, 0, None) == 1   # output dtype
    assert g(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 128, 128, 128, 1, None) == 1   # accumulate needs FP32
    assert g(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 0, 128, 128, 0, 0, None) == 2     # K == 0
    assert g(FAKE + 4, FAKE, FAKE, FAKE, 0, FAKE, 0, 128, 128, 128, 0, None) == 3
    assert g(None, FAKE, FAKE, FAKE, 0, FAKE, 0, 128, 128, 128, 0, None) == 1
    assert g(None, None, None, None, 0, None, 0, 0, 128, 128, 0, None) == 0     # empty: no-op


@pytest.mark.parametrize("name", ["fp8bs_grouped_gemm", "fp8bs_grouped_gemm_pow2"])
def test_grouped_gemm_argument_errors(lib, name):
    g = getattr(lib, name)
    assert g(FAKE, FAKE, 256, FAKE, 0, FAKE, FAKE, FAKE, 0, 128, 128, None) == 1      # no groups
    assert g(FAKE, FAKE, 256, FAKE, 513, FAKE, FAKE, FAKE, 0, 128, 128, None) == 1
    assert g(FAKE, FAKE, 256, None, 2, FAKE, FAKE, FAKE, 0, 128, 128, None) == 1      # offsets missing
    assert g(FAKE, FAKE, 256, FAKE, 2, FAKE, FAKE, FAKE, 0, 128, 100, None) == 2
    assert g(FAKE, FAKE, 256, FAKE, 2, FAKE, FAKE, FAKE + 1, 0, 128, 128, None) == 3


def test_moe_row_kernels_argument_errors(lib):
    gq, gb, cb = lib.fp8bs_gather_q_rows, lib.fp8bs_gather_bf16_rows, lib.fp8bs_moe_combine
    assert gq(FAKE, FAKE, 10, 100, 0, FAKE, 10, FAKE, FAKE, 1, None) == 2      # H % 128
    assert gq(FAKE, FAKE, 10, 128, 2, FAKE, 10, FAKE, FAKE, 1, None) == 1      # unknown scale layout
    assert gq(FAKE, FAKE, 10, 128, 0, None, 10, FAKE, FAKE, 1, None) == 1      # no index
    assert gq(FAKE + 4, FAKE, 10, 128, 0, FAKE, 10, FAKE, FAKE, 1, None) == 3
    assert gq(None, None, 0, 128, 0, None, 0, None, None, 0, None) == 0        # empty: no-op
    assert gb(FAKE, 10, 12, FAKE, 10, FAKE, None) == 2                         # N % 8
    assert gb(FAKE, 10, 16, FAKE, 10, FAKE + 2, None) == 3
    assert cb(FAKE, 10, 16, FAKE, FAKE, 4, 0, FAKE, None) == 1                 # k < 1
    assert cb(FAKE, 10, 16, FAKE, FAKE, 4, 65, FAKE, None) == 1                # k > 64
    assert cb(FAKE, 10, 12, FAKE, FAKE, 4, 2, FAKE, None) == 2
    assert cb(FAKE, 10, 16, None, FAKE, 4, 2, FAKE, None) == 1
    sq = lib.fp8bs_scatter_q_rows
    #        q     s     rows_in H   lay pos   k  zero  nz rows_out q_out s_out lay
    assert sq(FAKE, FAKE, 10, 100, 0, FAKE, 2, None, 0, 20, FAKE, FAKE, 1, None) == 2    # H % 128
    assert sq(FAKE, FAKE, 10, 128, 0, FAKE, 0, None, 0, 20, FAKE, FAKE, 1, None) == 1    # k < 1
    assert sq(FAKE, FAKE, 10, 128, 0, FAKE, 65, None, 0, 20, FAKE, FAKE, 1, None) == 1   # k > 64
    assert sq(FAKE, FAKE, 10, 128, 0, FAKE, 2, None, -1, 20, FAKE, FAKE, 1, None) == 1   # n_zero < 0
    assert sq(FAKE, FAKE, 10, 128, 0, FAKE, 2, None, 3, 20, FAKE, FAKE, 1, None) == 1    # zero list missing
    assert sq(FAKE, FAKE, 10, 128, 3, FAKE, 2, None, 0, 20, FAKE, FAKE, 1, None) == 1    # unknown layout
    assert sq(FAKE, FAKE, 10, 128, 0, None, 2, None, 0, 20, FAKE, FAKE, 1, None) == 1    # no positions
    assert sq(FAKE, FAKE, 10, 128, 0, FAKE, 2, None, 0, 20, FAKE + 4, FAKE, 1, None) == 3
    assert sq(FAKE, FAKE, 2 ** 30, 128, 0, FAKE, 4, None, 0, 20, FAKE, FAKE, 1, None) == 2  # rows_in * k >= 2^31
    assert sq(FAKE, FAKE, 10, 128, 0, FAKE, 2, None, 0, 20, None, None, 0, None) == 1       # no output buffers
    assert sq(None, None, 0, 128, 0, None, 2, None, 0, 20, None, None, 0, None) == 0       # nothing to move
    assert sq(None, None, 0, 128, 0, None, 2, None, 0, 0, None, None, 0, None) == 0        # empty: no-op


def test_quantize_act_weight_argument_errors(lib):
    q = lib.fp8bs_quantize_act_weight
    ok = (FAKE, 128, 256, 256, FAKE, FAKE, FAKE, 128, 256, 256, FAKE, FAKE, 0, None)

    def call(**kw):
        names = ["x", "M", "K", "ldx", "xq", "sx", "w", "N", "Kw", "ldw", "wq", "sw", "mode", "stream"]
        args = dict(zip(names, ok))
        args.update(kw)
        return q(*[args[n] for n in names])
    assert call(K=100, ldx=100) == 2                 # K % 128
    assert call(N=100) == 2                          # N % 128
    assert call(Kw=100, ldw=100) == 2                # Kw % 128
    assert call(ldx=128) == 1                        # ldx < K
    assert call(ldw=128) == 1                        # ldw < Kw
    assert call(mode=7) == 1                         # scale mode
    assert call(x=None) == 1
    assert call(sw=None) == 1
    assert call(wq=FAKE + 8) == 3
    assert call(ldx=260) == 3                        # ldx * 2 not a multiple of 16
    assert call(M=-1) == 1
    assert call(x=None, xq=None, sx=None, M=0, w=None, wq=None, sw=None, N=0) == 0   # both empty: no-op


def test_diag_unpromoted_argument_errors(lib):
    g = lib.fp8bs_diag_gemm_unpromoted
    assert g(FAKE, FAKE, FAKE, 128, 256, 100, None) == 2    # K % 128
    assert g(FAKE, FAKE, FAKE, 128, 128, 128, None) == 2    # N % 256
    assert g(FAKE, FAKE, FAKE, 100, 256, 128, None) == 2    # M % 128
    assert g(FAKE, FAKE, FAKE, 128, 256, 0, None) == 2      # K == 0
    assert g(FAKE, FAKE, FAKE, -128, 256, 128, None) == 1
    assert g(None, FAKE, FAKE, 128, 256, 128, None) == 1
    assert g(FAKE, FAKE, FAKE + 4, 128, 256, 128, None) == 3
    assert g(None, None, None, 0, 256, 128, None) == 0     # empty: no-op


def test_selftest_argument_errors(lib):
    assert lib.fp8bs_selftest_wait_timeout(0, None) == 1
    assert lib.fp8bs_selftest_wait_timeout(20000000, None) == 1


def test_timeout_setting(lib):
    assert lib.fp8bs_set_wait_timeout_ms(-1) == 1
    assert lib.fp8bs_set_wait_timeout_ms(500) == 0
    assert lib.fp8bs_set_wait_timeout_ms(0) == 0


def test_missing_library_fails_loudly(tmp_path):
    import importlib
    mod = importlib.import_module("fp8_fine_grained_fp8bs_gb300")
    with pytest.raises(RuntimeError):
        saved = mod._lib
        mod._lib = None
        try:
            mod.load_library(str(tmp_path / "nope.so"))
        finally:
            mod._lib = saved
