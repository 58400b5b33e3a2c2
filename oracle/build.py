"""Compile the C oracle into a shared library (test infrastructure only).

``build()`` is called by the tests and by the package build step; it is a
plain ``gcc`` invocation with no link to the CUDA library.  ``-ffp-contract=off``
keeps fp64 rounding identical on x86_64 and aarch64 hosts.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mk_oracle.c")
OUT = os.path.join(HERE, "_build", "libmk_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(src: str = SRC, out: str = OUT, force: bool = False, quiet: bool = True) -> str:
    """Compile ``src`` to ``out`` unless ``out`` is newer than its sources."""
    hdr = os.path.join(os.path.dirname(os.path.abspath(src)), "mk_oracle.h")
    deps = [src] + ([hdr] if os.path.exists(hdr) else [])
    if not force and os.path.exists(out) and all(os.path.getmtime(out) >= os.path.getmtime(d) for d in deps):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-I", os.path.dirname(os.path.abspath(src)), "-I", HERE, "-o", tmp, src, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + " ".join(cmd) + "\n" + res.stderr)
    if not quiet and res.stderr:
        sys.stderr.write(res.stderr)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, quiet=False))
