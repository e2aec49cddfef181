"""Build the CUDA library in-tree: ``io_aware_attention_fa2_gb300/_build/libfa_gb300.so``.

nvcc compiles each translation unit for sm_103a only (``-gencode arch=compute_103a,
code=sm_103a``), in parallel, and links them into one shared library with the CUDA runtime
linked statically, so the library needs no CUDA shared object besides the driver at run time.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
CSRC = os.path.join(_PKG, "csrc")
INCLUDE = os.path.join(_ROOT, "include")
BUILD_DIR = os.path.join(_PKG, "_build")
LIB = os.path.join(BUILD_DIR, "libfa_gb300.so")

SOURCES = ["fa_fwd_kernel.cu", "fa_bwd_kernel.cu", "fa_api.cpp", "fa_noalloc.cu"]
HEADERS = ["fa_internal.h", "ptx_sm103.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise FileNotFoundError("nvcc not found")


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
    lang = ["-x", "cu"] if src.endswith(".cu") else []
    cmd = [nvcc(), *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC, *extra, *lang, "-c", os.path.join(CSRC, src), "-o", obj]
    subprocess.run(cmd, check=True)
    return obj


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(INCLUDE, "fa.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, extra_flags: list[str] | None = None, verbose: bool = False) -> str:
    """Compile and link the library if any source changed. Returns its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = list(extra_flags or [])
    if verbose:
        extra += ["-Xptxas", "-v"]
    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as pool:
        objs = list(pool.map(lambda s: _compile(s, extra), SOURCES))
    tmp = LIB + ".tmp%d" % os.getpid()
    subprocess.run([nvcc(), *ARCH, "-shared", "-cudart", "static", "-Xcompiler", "-fPIC",
                    *objs, "-o", tmp], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
