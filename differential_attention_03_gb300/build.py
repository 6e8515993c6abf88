"""Build libdiffattn.so in-tree with nvcc for sm_103a (GB300).

Every translation unit compiles in parallel; the shared library links the
CUDA runtime statically, so the only run-time dependency is the driver.
Usage: ``python -m differential_attention_03_gb300.build [--force]``.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdiffattn.so")
# The bounds-check build (-DDIFFATTN_BOUNDS): every TMA coordinate, tensor-memory
# address and global store of the kernels checked before the access; loaded
# instead of LIB when DIFFATTN_DEBUG=1.
BOUNDS_BUILD_DIR = os.path.join(PKG, "_build_bounds")
BOUNDS_LIB = os.path.join(PKG, "libdiffattn_bounds.so")

SOURCES = ["api.cu", "k_simt.cu", "k_twopass_v1_d128.cu", "k_onepass_v1_d64.cu", "k_onepass_v2_d128.cu",
           "k_decode.cu", "k_backward.cu", "k_gemm.cu",
           "k_twopass_v1_d128_f8.cu", "k_onepass_v2_d128_f8.cu", "k_onepass_v1_d64_f8.cu", "k_onepass_save.cu", "k_bwd_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (CUDA 13 toolkit required)")
    return cand


def _inputs():
    return (glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h"))
            + [os.path.abspath(__file__)])


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False, bounds: bool = False) -> str:
    """Compile and link libdiffattn.so (bounds=True: libdiffattn_bounds.so); returns its path."""
    lib, build_dir = (BOUNDS_LIB, BOUNDS_BUILD_DIR) if bounds else (LIB, BUILD_DIR)
    if not force and up_to_date(lib):
        return lib
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    if bounds:
        extra = extra + ["-DDIFFATTN_BOUNDS"]

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_verbose:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv,
                bounds="--bounds" in sys.argv))
