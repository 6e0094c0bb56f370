"""In-tree build of libgdr.so (sm_103a) with nvcc: one object per .cu file, compiled in parallel,
then linked into gated_delta_rule_prefill_gb300/libgdr.so.  No cmake, no torch extension."""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgdr.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def cflags(extra=()):
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler",
                    "-Wall", "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if os.environ.get("GDR_PTXAS_VERBOSE"):
        flags += ["-Xptxas", "-v"]
    return flags + list(extra)


def _compile(src: str) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    deps = [src, os.path.join(ROOT, "include", "gdr.h")] + glob.glob(os.path.join(CSRC, "*.cuh"))
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(d) for d in deps):
        return obj
    tmp = obj + ".tmp%d" % os.getpid()
    r = subprocess.run([nvcc(), "-c", src, "-o", tmp] + cflags(), capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
    if r.stderr.strip() and os.environ.get("GDR_PTXAS_VERBOSE"):
        print(r.stderr)
    os.replace(tmp, obj)
    return obj


def build_library(force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    if force:
        for o in glob.glob(os.path.join(BUILD, "*.o")):
            os.remove(o)
    with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(_compile, srcs))
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(o) for o in objs)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    r = subprocess.run([nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs,
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True))
