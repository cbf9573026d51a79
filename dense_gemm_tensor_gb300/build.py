"""Builds the CUDA library ``libdgt_gemm.so`` in-tree with nvcc for sm_103a.

The translation units compile in parallel into ``_build/`` and link into
``dense_gemm_tensor_gb300/libdgt_gemm.so`` (CUDA runtime linked statically, so
the library loads on a machine without a GPU driver). A rebuild happens only
when a source or header is newer than the library.
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libdgt_gemm.so")
# The checked build: every range check in the kernels compiled in (DGT_CHECKED=1).
LIB_CHECKED = os.path.join(PKG, "libdgt_gemm_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# --compress-mode=size: the fatbinaries' device code compressed for size (the
# library is about a tenth as large; the code is unpacked once, when its module loads).
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "--compress-mode=size", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                     "-Xcompiler", "-Wall", "-Xcompiler", "-Wextra", "-Xcompiler", "-Wno-unused-parameter",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdgt_gemm.so")
    return path


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False, checked: bool = False) -> str:
    """Compile and link the library (``checked``: the range-checked debug
    build, ``libdgt_gemm_checked.so``); returns its path."""
    lib = LIB_CHECKED if checked else LIB
    if not force and up_to_date(lib):
        return lib
    bdir = os.path.join(BUILD, "checked") if checked else BUILD
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    if checked:
        extra += ["-DDGT_CHECKED=1"]

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src).replace(".cu", ".o"))
        cmd = [cc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_verbose:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv,
                checked="--checked" in sys.argv))
