"""Build the CSA / HCA kernel library for sm_103a, in-tree.

    python -m compressed_sparse_long_05_b300.build

compiles csrc/csa_lib.cu (one translation unit that includes every kernel)
into compressed_sparse_long_05_b300/lib/libcsa_b300.so with nvcc.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libcsa_b300.so")
LIB_TRACE = os.path.join(LIBDIR, "libcsa_b300_trace.so")   # phase-trace variant (-DCSA_TRACE)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the CSA kernels")


def sources():
    return sorted(os.path.join(SRC, f) for f in os.listdir(SRC) if f.endswith((".cu", ".cuh")))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    hdr = os.path.join(os.path.dirname(HERE), "include", "csa.h")
    return all(os.path.getmtime(s) <= t for s in sources() + [hdr, __file__])


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> str:
    """Compiles the library (or, with trace=True, its phase-trace variant)."""
    lib = LIB_TRACE if trace else LIB
    if not force and up_to_date(lib):
        return lib
    os.makedirs(LIBDIR, exist_ok=True)
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "--expt-relaxed-constexpr", "-Xptxas", "-v" if verbose else "-O3",
           *(["-DCSA_TRACE"] if trace else []), "-o", tmp, os.path.join(SRC, "csa_lib.cu")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if verbose:
        sys.stderr.write(res.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, trace="--trace" in sys.argv))
