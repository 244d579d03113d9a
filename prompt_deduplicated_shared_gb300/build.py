"""Build libzr.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under csrc/ is compiled in parallel; the objects are
linked into prompt_deduplicated_shared_gb300/libzr.so with the CUDA runtime
linked statically.  Re-running only recompiles sources newer than their object.

build(debug_bounds=True) makes the debug variant libzr_debug.so (objects in
_build_debug): every global index that a kernel derives from the device-built
plans is checked before the access, and a failed check records its site in
the status words (reported by zr_check_status) instead of touching memory.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libzr.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libzr_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc_path():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_mtime():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs.append(os.path.join(INCLUDE, "zr.h"))
    return max(os.path.getmtime(h) for h in hs)


def build(verbose: bool = False, force: bool = False, extra_flags=None, debug_bounds: bool = False) -> str:
    nvcc = nvcc_path()
    bdir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug_bounds else (BUILD, LIB)
    os.makedirs(bdir, exist_ok=True)
    hdr_t = _headers_mtime()
    flags = NVCC_FLAGS + (["-DZR_DEBUG_BOUNDS"] if debug_bounds else []) + list(extra_flags or [])
    jobs = []
    objs = []
    for src in _sources():
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(src), hdr_t):
            jobs.append([nvcc, *ARCH, *flags, "-c", src, "-o", obj])

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {cmd[-3]}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(run, jobs))
    if jobs or not os.path.exists(lib):
        link = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", lib + ".tmp", *objs, "-ldl"]
        run(link)
        os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
