"""In-tree build of libspecverify.so (CUDA kernels for sm_103a + the C ABI).

Seven compilation units, one -gencode, compiled in parallel and linked with the
shared cudart (so the process keeps a single CUDA runtime with PyTorch): the
host side (csrc/spec_verify.cu) and six groups of kernels (csrc/kernel_unit.cu
with SPECV_UNIT = 1..6; both include csrc/spec_kernels.cuh).  The library is
written next to this file.
"""
from __future__ import annotations

import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
HDR = os.path.join(ROOT, "include", "spec_verify.h")
LIB = os.path.join(PKG, "libspecverify.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMPILE_FLAGS = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC"]
LINK_FLAGS = [*ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
# (source, extra defines); the heaviest units first, so they start first
UNITS = [("kernel_unit.cu", ["-DSPECV_UNIT=%d" % u]) for u in (6, 5, 2, 1, 4, 3)] + [("spec_verify.cu", [])]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def sources():
    return [HDR, __file__] + sorted(glob.glob(os.path.join(CSRC, "*.cu*"))) + \
        sorted(glob.glob(os.path.join(CSRC, "*.h")))


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in sources())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if it is missing or older than its sources."""
    if force or needs_build():
        tag = ".%d" % os.getpid()
        objs, procs = [], []
        try:
            for i, (src, defs) in enumerate(UNITS):
                obj = os.path.join(CSRC, "unit%d%s.o" % (i, tag))
                cmd = [nvcc(), *COMPILE_FLAGS, *defs, "-I", os.path.join(ROOT, "include"), "-c", "-o", obj,
                       os.path.join(CSRC, src)]
                if verbose:
                    print(" ".join(cmd), flush=True)
                procs.append(subprocess.Popen(cmd))
                objs.append(obj)
            codes = [p.wait() for p in procs]
            if any(codes):
                raise subprocess.CalledProcessError(max(codes), "nvcc")
            tmp = LIB + ".tmp" + tag
            cmd = [nvcc(), *LINK_FLAGS, "-o", tmp, *objs]
            if verbose:
                print(" ".join(cmd), flush=True)
            subprocess.check_call(cmd)
            os.replace(tmp, LIB)
        finally:
            for p in procs:
                if p.poll() is None:
                    p.kill()
            for o in objs:
                if os.path.exists(o):
                    os.remove(o)
    return LIB
