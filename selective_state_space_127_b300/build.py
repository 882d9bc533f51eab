"""Build libssmscan.so in-tree with nvcc for sm_103a (B300).

    python -m selective_state_space_127_b300.build [--force] [--debug-checks]

Sources: csrc/*.cu; public header: include/ssmscan.h. --debug-checks builds
libssmscan_debug.so instead, whose kernels check every computed global-memory index (a failed
check sets SSM_ERR_BOUNDS in the call's status word and skips the access). The CUDA runtime is linked
statically, so the library loads on a machine without a GPU (calls then fail with
SSM_ERR_CUDA) and needs no libcudart on the library path.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libssmscan.so")
DEBUG_LIB_PATH = os.path.join(PKG, "libssmscan_debug.so")
BUILD_DIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: set NVCC or put the CUDA toolkit on PATH")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date(lib: str = LIB_PATH) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, debug_checks: bool = False) -> str:
    """Compile every csrc/*.cu to an object (in parallel) and link libssmscan.so; with
    debug_checks, the index-checking build libssmscan_debug.so (-DSSM_DEBUG_CHECKS)."""
    lib = DEBUG_LIB_PATH if debug_checks else LIB_PATH
    if not force and up_to_date(lib):
        return lib
    nvcc = _nvcc()
    bdir = os.path.join(BUILD_DIR, "debug") if debug_checks else BUILD_DIR
    os.makedirs(bdir, exist_ok=True)
    extra = ["-DSSM_DEBUG_CHECKS"] if debug_checks else []
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd))
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        text = out.decode(errors="replace")
        if pr.returncode != 0:
            failed.append(f"{src}:\n{text}")
        elif verbose and text.strip():
            print(text)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    subprocess.check_call(cmd)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug_checks="--debug-checks" in sys.argv))
