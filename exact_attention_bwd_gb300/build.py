"""Builds libfa_gb300.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each CUDA source compiles to an object under ``_build/`` in parallel, then one link
step makes the shared library next to this file.  A rebuild happens only when a
source or header is newer than the library.

``build(trace=True)`` makes the separate trace library ``libfa_gb300_trace.so`` (objects
under ``_build_trace/``), compiled with -DFA_TRACE=1: its tensor-core kernels record
per-role event traces into the workspace (see csrc/trace.cuh and trace.py).  The product
library never contains the trace code.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(HERE, "libfa_gb300.so")
BUILD_DIR = os.path.join(HERE, "_build")
TRACE_LIB = os.path.join(HERE, "libfa_gb300_trace.so")
TRACE_BUILD_DIR = os.path.join(HERE, "_build_trace")
SOURCES = ["api.cu", "fwd.cu", "fwd256.cu", "fwd_e4m3.cu", "bwd.cu", "decode.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
                f"-I{INCLUDE}"]
# extra nvcc flags for tuning builds (e.g. -DFA_FWD_EXP_POLY_PAIRS=2); empty by default
EXTRA = os.environ.get("FA_NVCC_EXTRA", "").split()


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libfa_gb300.so")
    return exe


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    files += glob.glob(os.path.join(INCLUDE, "*.h"))
    return files


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> str:
    lib = TRACE_LIB if trace else LIB
    bdir = TRACE_BUILD_DIR if trace else BUILD_DIR
    if not force and not stale(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    defs = ["-DFA_TRACE=1"] if trace else []

    def one(src):
        obj = os.path.join(bdir, os.path.splitext(src)[0] + ".o")
        cmd = [cc] + FLAGS + defs + EXTRA + (["-Xptxas", "-v"] if verbose else []) + \
            ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(one, SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, trace="--trace" in sys.argv))
