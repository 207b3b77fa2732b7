"""Build libmattn.so (and libmattn_debug.so) in-tree with nvcc for sm_103a.

Usage: python -m block_sparse_attention_masked_gb300.build [--verbose] [--no-debug]
The libraries land next to this file; they are git-ignored and rebuilt on
every machine (the x86 build here and the aarch64 build on the GPU host
are not interchangeable).  libmattn_debug.so is the same sources compiled
with MATTN_DEBUG=1: device-side bounds checks on every TMA coordinate, work
item, key-tile entry, explicit-order value and decode ring slot, reported
through the device error word (MATTN_ERR_BOUNDS) instead of a fault.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libmattn.so")
DEBUG_LIB = os.path.join(PKG, "libmattn_debug.so")
BUILD_DIR = os.path.join(PKG, "_build")

SOURCES = ["attention_fwd.cu", "attention_persist.cu", "attention_sp.cu", "rr_select.cu", "received.cu", "decode.cu", "mattn_api.cpp",
           "mattn_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")
    return cand


def _compile(src: str, verbose: bool, debug: bool = False) -> str:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ("_debug.o" if debug else ".o"))
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj, "-std=c++17", "-O3", "-lineinfo",
           "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC, f"-DMATTN_DEBUG={1 if debug else 0}"] + ARCH
    if src.endswith(".cu"):
        cmd += ["--expt-relaxed-constexpr"]
        if verbose:
            cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    if verbose and (res.stdout or res.stderr):
        print(res.stdout + res.stderr, file=sys.stderr)
    return obj


def _link(objs, lib: str) -> None:
    tmp = lib + ".tmp"
    cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)


def build(verbose: bool = False, debug: bool = True) -> str:
    """Compiles every source (twice with `debug`: product and debug objects,
    all in parallel) and links libmattn.so and libmattn_debug.so."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    jobs = [(s, False) for s in SOURCES] + ([(s, True) for s in SOURCES] if debug else [])
    with ThreadPoolExecutor(max_workers=min(len(jobs), max(4, os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda j: _compile(j[0], verbose, j[1]), jobs))
    _link(objs[:len(SOURCES)], LIB)
    if debug:
        _link(objs[len(SOURCES):], DEBUG_LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="--verbose" in sys.argv, debug="--no-debug" not in sys.argv))
