"""Compile the CUDA sources into the in-tree shared library ``lib/libridgefill.so``.

Each ``csrc/*.cu`` file is compiled for sm_103a in parallel, then linked with
the static CUDA runtime (so the library loads without a GPU driver present).
``build(debug=True)`` makes ``lib/libridgefill_debug.so`` from the same sources
with ``RF_DEBUG=1``: every plain global store of the kernels is checked against
its buffer's extent (a store outside is skipped and reported through the device
error word) and every workspace region is followed by a guard band that each
call fills first and checks last.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from typing import List

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libridgefill.so")
LIB_DEBUG = os.path.join(LIBDIR, "libridgefill_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
    "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC,
]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found; the RidgeFill CUDA library cannot be built")
    return p


def sources() -> List[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _digest(flags: List[str]) -> str:
    h = hashlib.sha256()
    for f in sorted(os.listdir(CSRC)) + ["ridgefill.h"]:
        path = os.path.join(CSRC, f) if f != "ridgefill.h" else os.path.join(INCLUDE, f)
        with open(path, "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    h.update(" ".join(flags).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Build (if stale) and return the path of ``libridgefill.so`` (or, with ``debug``,
    of ``libridgefill_debug.so``)."""
    flags = NVCC_FLAGS + (["-DRF_DEBUG=1"] if debug else [])
    lib = LIB_DEBUG if debug else LIB
    objdir = BUILD + ("_debug" if debug else "")
    os.makedirs(objdir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    stamp = lib[:-3] + ".sha256"
    dig = _digest(flags)
    if not force and os.path.exists(lib) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == dig:
                return lib
    cc = nvcc()
    srcs = sources()

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    cmd = [cc] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "--cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(dig)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
    print(build(force=True, verbose=True, debug=True))
