"""In-tree build of the CUDA library ``_lib/libpa_verify.so`` for sm_103a.

Each translation unit is compiled by its own nvcc process (in parallel) and
then linked into one shared library with the CUDA runtime linked statically,
so loading it needs no CUDA toolkit on the library path.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "_lib")
OBJDIR = os.path.join(LIBDIR, "obj")
LIB = os.path.join(LIBDIR, "libpa_verify.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
SOURCES = ["pa_capi.cpp", "pa_split_bf16.cu", "pa_split_fp8.cu", "pa_combine.cu", "pa_kv_write.cu", "pa_verdict.cu", "pa_tc_split.cu", "pa_tc_split_d256.cu", "pa_tc_split_d64.cu", "pa_static.cu", "pa_dyn_plan.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpa_verify.so")
    return cand


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "pa_verify.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str) -> str:
    obj = os.path.join(OBJDIR, os.path.splitext(src)[0] + ".o")
    # -fno-gnu-unique: the launchers' per-device "attribute set" flags are function-local statics of template
    # instances; as GNU-unique symbols they would be shared with any other copy of this library loaded in the
    # same process, whose kernels would then launch without their shared-memory limit raised.
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fno-gnu-unique", "-I", INCLUDE,
           "-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cpp"):
        cmd[1:1] = ["-x", "cu"]
    subprocess.run(cmd, check=True)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles the library if any source is newer than it; returns its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(_compile, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}")
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True)
