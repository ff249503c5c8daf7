"""Build libjt.so (the CUDA kernels + C ABI) in-tree for sm_103a.

Each .cu file is compiled by nvcc in parallel, then linked into a shared
library with the CUDA runtime linked statically (no libcudart.so needed at
load time; the driver is reached lazily).  Usage: ``python -m
tree_speculative_decoding_jt_gb300.build [--force] [--variant checks]`` or
``build()`` from Python.

Variants: the default library, and ``checks`` (libjt_checks.so), built with
-DJT_CHECKS (extra device-side validation of input contents; a failed check
sets the workspace error word, it never traps) and -DJT_NVTX (an NVTX range
around every entry point).  The binding loads the checks variant when the
environment variable JT_LIB_VARIANT=checks is set.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libjt.so")
BUILD_DIR = os.path.join(HERE, "_build")
VARIANTS = {"": [], "checks": ["-DJT_CHECKS", "-DJT_NVTX"]}


def lib_path(variant: str = "") -> str:
    if variant not in VARIANTS:
        raise ValueError(f"unknown libjt variant {variant!r} (known: {sorted(VARIANTS)})")
    return LIB if not variant else os.path.join(HERE, f"libjt_{variant}.so")
SOURCES = ["jt_api.cu", "tree_build.cu", "verify_accept.cu", "tree_attn.cu", "tree_attn_f32.cu", "jt_noalloc.cu", "verify_stochastic.cu", "jt_selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libjt")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(HERE, "..", "include", "jt.h"))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant: str = "") -> str:
    lib = lib_path(variant)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    bdir = BUILD_DIR + (f"_{variant}" if variant else "")
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    flags = [*FLAGS, *VARIANTS[variant], *extra_flags]

    def compile_one(src):
        obj = os.path.join(bdir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    v = sys.argv[sys.argv.index("--variant") + 1] if "--variant" in sys.argv else ""
    print(build(force="--force" in sys.argv, verbose=True, variant=v))
