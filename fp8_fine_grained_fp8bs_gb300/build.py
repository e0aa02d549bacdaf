"""Builds the CUDA library ``_build/libfp8bs.so`` in-tree with nvcc.

One ``-gencode`` (sm_103a), the translation units compiled in parallel,
then linked into a shared library that exports only the ``fp8bs_*`` C ABI.
The CUDA runtime is linked statically and bound symbolically, so the
library never resolves runtime calls against another copy of the runtime
loaded in the same process.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libfp8bs.so")

SOURCES = ["api.cu", "quantize.cu", "gemm.cu", "gemm_mx.cu", "moe.cu", "diag.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build fp8bs")
    return cand


def _inputs_newer_than(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "fp8bs.h"), __file__]
    return any(os.path.getmtime(p) > t for p in deps)


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles (if needed) and returns the path of libfp8bs.so."""
    if not force and not _inputs_newer_than(LIB_PATH):
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    log = "".join(f"== {s}\n{out}" for s, (_, out) in zip(SOURCES, results))
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as f:
        f.write(log)
    if verbose:
        sys.stdout.write(log)
    version_script = os.path.join(BUILD_DIR, "exports.map")
    with open(version_script, "w") as f:
        f.write("{ global: fp8bs_*; local: *; };\n")
    tmp = LIB_PATH + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results],
           "-Xlinker", "-Bsymbolic", "-Xlinker", f"--version-script={version_script}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
