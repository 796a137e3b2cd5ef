"""Builds libgma.so in-tree with nvcc for sm_103a (no cmake, no torch extension machinery).

Each .cu translation unit is compiled in parallel, then linked into
``gaussian_mixture_sequence_gma_gb300/_lib/libgma.so``.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libgma.so")
# bounds-check debug build: the same sources with -DGMA_BOUNDS_CHECK (see gma_debug_bounds_read)
LIB_CHECKED = os.path.join(OUT_DIR, "libgma_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found")
    return p


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, checked: bool = False) -> str:
    """libgma.so, or (checked) its bounds-check debug variant libgma_checked.so."""
    srcs = sources()
    headers = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    obj_dir = os.path.join(OUT_DIR, "obj_checked" if checked else "obj")
    lib = LIB_CHECKED if checked else LIB
    extra = ["-DGMA_BOUNDS_CHECK"] if checked else []
    os.makedirs(obj_dir, exist_ok=True)
    procs = []
    objs = []
    for s in srcs:
        o = os.path.join(obj_dir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or _stale(o, [s] + headers + [__file__]):
            cmd = [nvcc()] + ARCH + FLAGS + extra + (["-Xptxas", "-v"] if ptxas_info else []) + ["-c", s, "-o", o]
            procs.append((s, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for s, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0 or ptxas_info:
            sys.stdout.write(out)
        if p.returncode != 0:
            failed.append(s)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    if force or procs or _stale(lib, objs):
        tmp = lib + ".tmp%d" % os.getpid()
        # shared cudart: the library joins the CUDA runtime the host process (e.g. torch) already uses,
        # so the current device and stream handles are the same on both sides of the ABI
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-Xlinker", "-rpath=/usr/local/cuda/lib64",
                                 "-o", tmp] + objs + ["-lcublasLt"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> list[str]:
    """libgma.so and libgma_checked.so, their translation units compiled concurrently."""
    import concurrent.futures as cf
    with cf.ThreadPoolExecutor(2) as ex:
        futs = [ex.submit(build, force, False, False, checked) for checked in (False, True)]
        return [f.result() for f in futs]


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                checked="--checked" in sys.argv))
