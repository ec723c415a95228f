"""Builds libtkv.so in-tree for GB300 (sm_103a) with nvcc.

The translation units are compiled in parallel and linked into one shared
library next to this file; nothing is installed anywhere else. build(debug=True)
makes libtkv_debug.so instead: the same sources with TKV_DEBUG defined, which
turns on the kernels' device index checks (selected at run time by
TKV_LIB=debug).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(HERE, "libtkv.so")
LIB_DEBUG = os.path.join(HERE, "libtkv_debug.so")
SOURCES = ["attention.cu", "classify.cu", "movement.cu", "runtime.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtkv.so")
    return cand


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, debug: bool = False) -> str:
    nvcc = _nvcc()
    out_dir = os.path.join(BUILD, "debug") if debug else BUILD
    lib = LIB_DEBUG if debug else LIB
    flags = FLAGS + (["-DTKV_DEBUG"] if debug else [])
    os.makedirs(out_dir, exist_ok=True)
    headers = [os.path.join(CSRC, "tkv_internal.h"), os.path.join(INCLUDE, "tkv.h")]
    jobs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(out_dir, s.replace(".cu", ".o"))
        if force or _stale(obj, [src] + headers):
            jobs.append([nvcc, *ARCH, *flags, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        if verbose:
            sys.stderr.write(r.stdout + r.stderr)

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(run, jobs))
    objs = [os.path.join(out_dir, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or _stale(lib, objs):
        run([nvcc, *ARCH, "-shared", "-o", lib, *objs, "-lcudart"])
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug="--debug" in sys.argv))
