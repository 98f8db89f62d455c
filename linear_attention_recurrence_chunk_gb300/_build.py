"""In-tree build of the CUDA library ``libkda_gb300.so`` for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled by its own ``nvcc`` process (in
parallel), then linked into one shared library beside this file.  No cmake,
no torch extension machinery: the library is plain C ABI (``include/kda.h``).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libkda_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fvisibility=hidden"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkda_gb300.so")
    return cand


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link the library if any source is newer than it.  Returns its path."""
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    tmpdir = tempfile.mkdtemp(prefix="kda_build_", dir=PKG)
    try:
        flags = ARCH + NVCC_FLAGS + ["-I", INCLUDE, "-I", CSRC]
        if ptxas_info:
            flags += ["-Xptxas", "-v"]

        def compile_one(src):
            obj = os.path.join(tmpdir, os.path.basename(src) + ".o")
            r = subprocess.run([nvcc, *flags, "-c", src, "-o", obj], capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
            if verbose or ptxas_info:
                print(r.stderr, end="")
            return obj

        srcs = sources()
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
            objs = list(ex.map(compile_one, srcs))
        tmp_lib = os.path.join(tmpdir, "libkda_gb300.so")
        r = subprocess.run([nvcc, *ARCH, "-shared", *objs, "-o", tmp_lib], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp_lib, LIB)
    finally:
        shutil.rmtree(tmpdir, ignore_errors=True)
    return LIB


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv))
