"""Build the CUDA library ``_build/libmk.so`` for sm_103a with nvcc.

Two translation units (device code, host API) compile in parallel, then link
into one shared library with the CUDA runtime linked statically.  The
library's ABI is ``include/mk.h``.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libmk.so")
UNITS = ["mk_kernels.cu", "mk_api.cu", "mk_noalloc.cu"]

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _deps():
    return (glob.glob(os.path.join(CSRC, "*")) + [os.path.join(INCLUDE, "mk.h"), os.path.abspath(__file__)])


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of ``libmk.so``."""
    if not force and os.path.exists(LIB):
        t = os.path.getmtime(LIB)
        if all(os.path.getmtime(d) <= t for d in _deps()):
            return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    procs = []
    objs = []
    for u in UNITS:
        obj = os.path.join(OUT_DIR, u.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [NVCC, *ARCH, *FLAGS, "-c", os.path.join(CSRC, u), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    for cmd, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + out)
        if verbose and out:
            print(out, file=sys.stderr)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
