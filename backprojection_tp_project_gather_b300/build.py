"""Build libtp_b300.so (the C-ABI library) in-tree with nvcc for sm_103a.

Usage: ``python -m backprojection_tp_project_gather_b300.build [-v]``.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libtp_b300.so")
LIB_DEBUG = os.path.join(HERE, "libtp_b300_debug.so")   # -DTP_DEBUG_BOUNDS: index checks
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-Wall", "-shared",
         "--expt-relaxed-constexpr"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
    deps.append(os.path.join(HERE, "..", "include", "tp.h"))
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Build the library (debug: the bounds-checking variant, libtp_b300_debug.so)."""
    lib = LIB_DEBUG if debug else LIB
    if not force and not _stale(lib):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, *FLAGS, *(["-DTP_DEBUG_BOUNDS"] if debug else []),
           *(["-Xptxas", "-v"] if verbose else []), "-o", tmp, *sources()]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    if verbose:
        sys.stderr.write(r.stdout + r.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
