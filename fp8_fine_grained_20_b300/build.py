"""Build ``libfp8fg.so`` (the C-ABI CUDA library) in-tree for sm_103a.

Usage: ``python -m fp8_fine_grained_20_b300.build [--force] [--verbose]``.
nvcc cross-compiles without a GPU, so this runs on any machine with CUDA 13.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libfp8fg.so")
# the same library with every device write bounds-checked (-DFP8FG_BOUNDS): a
# debug build, loaded instead of LIB when FP8FG_BOUNDS=1 is set
LIB_BOUNDS = os.path.join(HERE, "libfp8fg_bounds.so")
SOURCES = [os.path.join(CSRC, "fp8fg.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("ptx.cuh", "quant.cuh", "gemm.cuh", "gemm_mx.cuh", "swiglu.cuh", "probe.cuh")] + [
    os.path.join(ROOT, "include", "fp8fg.h")]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-std=c++17", "-lineinfo",
    "-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-fmad=true",
    "-Xcompiler", "-fPIC", "-shared",
    "-I", os.path.join(ROOT, "include"),
]


def _stale(lib) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in DEPS)


def build(force: bool = False, verbose: bool = False, bounds: bool = False) -> str:
    """Compile the library (the bounds-checked debug build with bounds=True) if
    it is missing or older than its sources."""
    lib = LIB_BOUNDS if bounds else LIB
    if not force and not _stale(lib):
        return lib
    tmp = lib + ".tmp.%d" % os.getpid()
    cmd = [NVCC, *FLAGS, *(["-DFP8FG_BOUNDS"] if bounds else []), *(["-Xptxas", "-v"] if verbose else []),
           *SOURCES, "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        sys.stderr.write(res.stdout + res.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv, bounds="--bounds" in sys.argv))
