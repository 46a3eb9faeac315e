"""Builds libsparda.so in-tree from csrc/*.cu for sm_103a (GB300).

Each translation unit compiles in parallel with nvcc; the objects link into one shared
library with the CUDA runtime linked statically, so the library loads on a host without a
GPU driver (the driver is only needed once a call reaches the GPU).

    python -m block_sparse_attention_forecast_gb300.build [--force]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libsparda.so")
# the per-CTA timeline variant (-DSPARDA_TIMELINE): a separate library, never the product one
LIB_TIMELINE = os.path.join(OUT_DIR, "libsparda_timeline.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libsparda")
    return exe


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(ROOT, "include", "sparda.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib=LIB):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _compile(src, extra, tag=""):
    obj = os.path.join(OUT_DIR, os.path.basename(src) + tag + ".o")
    cmd = [nvcc()] + ARCH + FLAGS + extra + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    return obj, r.stderr


def build(force=False, verbose=False, extra=None, timeline=False):
    """Compile every CUDA source and link libsparda.so; returns the library path. timeline=True
    builds the per-CTA timeline variant (libsparda_timeline.so) instead."""
    extra = list(extra or [])
    lib, tag = (LIB_TIMELINE, ".tl") if timeline else (LIB, "")
    if timeline:
        extra.append("-DSPARDA_TIMELINE")
    if not force and (timeline or not extra) and up_to_date(lib):
        return lib
    os.makedirs(OUT_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        results = list(ex.map(lambda s: _compile(s, extra, tag), sources()))
    objs = [o for o, _ in results]
    if verbose:
        for _, err in results:
            if err.strip():
                print(err, file=sys.stderr)
    tmp = lib + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, lib)
    for o in objs:
        os.remove(o)
    return lib


if __name__ == "__main__":
    args = sys.argv[1:]
    print(build(force="--force" in args, verbose="-v" in args,
                extra=["-Xptxas", "-v"] if "--ptxas" in args else None))
