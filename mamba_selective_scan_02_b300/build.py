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
LIB_DEBUG = os.path.join(LIBDIR, "libssmscan_debug.so")   # -DSSM_DEBUG: index checks on every store
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


FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC"]


def nvcc_cmd(out: str, extra=()):
    """One nvcc call that compiles every source straight into the library."""
    return (["nvcc", *ARCH, *FLAGS, "-shared", "-I", os.path.join(ROOT, "include"), *extra, "-o", out]
            + sources())


def build(force: bool = False, verbose: bool = False, extra=(), jobs: int = 0, debug: bool = False) -> str:
    """Compile the library if any source is newer than it.  Returns its path.

    Each source compiles to its own object in a separate nvcc process (the
    files share no device code, only inline header functions), in parallel,
    and one nvcc call links them.  `debug` builds libssmscan_debug.so with
    -DSSM_DEBUG instead."""
    out = LIB_DEBUG if debug else LIB
    if debug:
        extra = (*extra, "-DSSM_DEBUG")
    if not force and not stale(out):
        return out
    from concurrent.futures import ThreadPoolExecutor
    os.makedirs(LIBDIR, exist_ok=True)
    tag = "%d%s" % (os.getpid(), "d" if debug else "")
    objdir = os.path.join(LIBDIR, "obj." + tag)
    os.makedirs(objdir, exist_ok=True)
    inc = ["-I", os.path.join(ROOT, "include")]
    srcs = sources()
    objs = [os.path.join(objdir, os.path.basename(src) + ".o") for src in srcs]
    cmds = [["nvcc", *ARCH, *FLAGS, *inc, *extra, "-c", src, "-o", obj] for src, obj in zip(srcs, objs)]
    if verbose:
        for c in cmds:
            print(" ".join(c), file=sys.stderr)
    workers = jobs or min(len(cmds), os.cpu_count() or 1)
    with ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), cmds))
    for c, r in zip(cmds, results):
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise subprocess.CalledProcessError(r.returncode, c)
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
    tmp = out + ".tmp" + tag
    subprocess.run(["nvcc", *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, out)
    for o in objs:
        os.remove(o)
    os.rmdir(objdir)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv,
                extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else ()))
