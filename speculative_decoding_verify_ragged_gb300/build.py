"""Build the in-tree CUDA library ``libsdv.so`` for sm_103a.

Each translation unit is compiled with nvcc in parallel, then linked into a
shared library next to this file (the CUDA runtime is linked statically).
Run ``python -m speculative_decoding_verify_ragged_gb300.build``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsdv.so")
BUILD_TRACE = os.path.join(HERE, "_build_trace")
LIB_TRACE = os.path.join(HERE, "libsdv_trace.so")
SOURCES = ("api.cu", "gemm.cu", "gemm_tc.cu", "gemm_tc_q4.cu", "gemm_q4.cu", "attention.cu", "attention_tc.cu", "step_kernels.cu", "noalloc.cu", "sched.cpp", "ngram.cpp")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                   "-I", os.path.join(ROOT, "include")] + list(extra)


def _compile(src: str, extra, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + (".cpp.o" if src.endswith(".cpp") else ".o"))
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj] + flags(extra)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(verbose: bool = False, extra=(), trace: bool = False) -> str:
    """Build libsdv.so; trace=True builds libsdv_trace.so instead, the same
    library with the step-timeline stamps compiled in (sdv_trace_enable)."""
    build_dir, lib = (BUILD_TRACE, LIB_TRACE) if trace else (BUILD, LIB)
    extra = tuple(extra) + (("-DSDV_TRACE",) if trace else ())
    os.makedirs(build_dir, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print(lib)
    return lib


if __name__ == "__main__":
    args = sys.argv[1:]
    build(verbose=True, extra=[a for a in args if a != "--trace"], trace="--trace" in args)
