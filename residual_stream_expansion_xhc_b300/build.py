"""Build the xHC CUDA library (libxhc.so) in-tree for sm_103a with nvcc."""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libxhc.so")
LIB_DEBUG = os.path.join(PKG, "libxhc_debug.so")   # -DXHC_DEBUG: bounds-checked streaming kernels
SOURCES = ["xhc_api.cu", "xhc_simt.cu", "xhc_bwd.cu", "xhc_tc.cu", "xhc_stream.cu", "xhc_gs.cu", "xhc_router.cu", "xhc_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(os.path.dirname(PKG), "include", "xhc.h"))
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile every CUDA source of the library into one shared object
    (debug: the bounds-checked build, libxhc_debug.so)."""
    lib = LIB_DEBUG if debug else LIB
    if not force and not _stale(lib):
        return lib
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-diag-suppress", "128", "-o", lib + ".tmp"]
    if debug:
        cmd += ["-DXHC_DEBUG"]
    cmd += [os.path.join(CSRC, s) for s in SOURCES]
    cmd += ["-lcuda"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
