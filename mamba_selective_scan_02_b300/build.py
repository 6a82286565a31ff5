"""In-tree build of libssmscan.so for sm_103a with nvcc (no JIT cache).

``python -m mamba_selective_scan_02_b300.build`` (or ``build()``) compiles every
``csrc/*.cu`` into ``mamba_selective_scan_02_b300/lib/libssmscan.so``.
"""

from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libssmscan.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def deps():
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + sorted(
        glob.glob(os.path.join(CSRC, "*.h"))) + [os.path.join(ROOT, "include", "ssm_scan.h")]


def stale(out: str = LIB) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(p) > t for p in deps())


def nvcc_cmd(out: str, extra=()):
    return (["nvcc", *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
             "-I", os.path.join(ROOT, "include"), *extra, "-o", out] + sources())


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile the library if any source is newer than it.  Returns its path."""
    if not force and not stale():
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = nvcc_cmd(tmp, extra)
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else ())
    print(LIB)
