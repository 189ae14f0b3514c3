"""Compile the CUDA library in place (nvcc, sm_103a only)."""
from __future__ import annotations

import os
import shutil
import subprocess
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, "zero_opt.cu"), os.path.join(CSRC, "ckpt.cpp"),
           os.path.join(CSRC, "noalloc.cu"), os.path.join(CSRC, "host_step.cpp")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("kernels.cuh", "zero_opt_internal.h",
                                                     "host_util.h", "decide_core.h", "host_cast.h")] + [
    os.path.join(INCLUDE, "zero_opt.h")]
LIB = os.path.join(PKG, "libzero_opt.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -fmad=false: no multiply-add contraction anywhere in device code, so the
# binary64 per-step scalars round exactly like the host definition; the
# per-element binary32 update uses explicit _rn intrinsics regardless.
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-fmad=false",
                     "-Xcompiler", "-fPIC,-O3,-ffp-contract=off,-fno-math-errno",
                     "-I", INCLUDE]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found")
    return path


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in DEPENDS)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and not stale():
        return LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=PKG)
    os.close(fd)
    cmd = [nvcc(), *NVCC_FLAGS, "-shared", "-o", tmp, *SOURCES]
    if ptxas_info:
        cmd.insert(1, "-Xptxas=-v")
    try:
        r = subprocess.run(cmd, check=True, capture_output=True, text=True)
        if verbose or ptxas_info:
            print(r.stdout + r.stderr)
        os.replace(tmp, LIB)
    except subprocess.CalledProcessError as e:
        if os.path.exists(tmp):
            os.unlink(tmp)
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + e.stderr) from e
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, ptxas_info="-v" in sys.argv))
