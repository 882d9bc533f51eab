"""Build and run the unit-rate microbenchmark (csrc/rates/unit_rates.cu) on GPU 0.

    python -m selective_state_space_127_b300.unit_rates [--build-only]

Prints one JSON object: lane operations per clock per SM for the SFU functions (ex2, lg2,
rcp, tanh), FP32 FMA (scalar and packed f32x2), shared-memory bytes delivered per clock by
load width and address sharing, warp shuffles, and multiply-adds per clock of the legacy
warp MMA. The selective scan's "alu" roofline (one ex2 and four FP32 lane operations per
state update) is taken from these rates.
"""
from __future__ import annotations

import os
import subprocess
import sys

from .build import ARCH, BUILD_DIR, CSRC, _nvcc

SRC = os.path.join(CSRC, "rates", "unit_rates.cu")
EXE = os.path.join(BUILD_DIR, "unit_rates")


def build() -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    if not os.path.exists(EXE) or os.path.getmtime(EXE) < os.path.getmtime(SRC):
        subprocess.check_call([_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", SRC, "-o", EXE])
    return EXE


def main() -> int:
    exe = build()
    if "--build-only" in sys.argv:
        print(exe)
        return 0
    return subprocess.call([exe])


if __name__ == "__main__":
    sys.exit(main())
