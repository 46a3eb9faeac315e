"""Diagnostic: throughput of back-to-back tcgen05.mma (bf16 -> fp32, M = 128) on this GPU for
the operand shapes of the prefill attention, from one issuing thread per SM.

    python -m block_sparse_attention_forecast_gb300.mma_rate

Compiles csrc/diag/mma_rate.cu (not part of libsparda) with nvcc into _lib/ and runs it.
"""
from __future__ import annotations

import os
import subprocess

from . import build


def main():
    src = os.path.join(build.CSRC, "diag", "mma_rate.cu")
    exe = os.path.join(build.OUT_DIR, "mma_rate")
    os.makedirs(build.OUT_DIR, exist_ok=True)
    cmd = [build.nvcc()] + build.ARCH + ["-O3", "-std=c++17", "-I" + os.path.join(build.ROOT, "include"), src, "-o", exe]
    subprocess.run(cmd, check=True)
    subprocess.run([exe], check=True)


if __name__ == "__main__":
    main()
